// Packing and reconstruction ("How Prompt Deduplication Works": "Creating
// Deduplicated Batch", "Reconstructing Original Batch", "Working with
// Packed/Unpacked Sequences").
//
// Every slot of the packed layout [Prompt_1][R_1_1]..[R_1_n][Prompt_2].. is a
// contiguous run of source rows, so both directions are lists of contiguous
// row-range copies ("segments").  One planning launch turns the grouping and
// the mask into slot offsets and three segment tables (pack, reconstruct, pad
// rows); the data movement is one generic kernel that streams each segment
// with 16-byte vector loads and stores.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <climits>

#include "zr_internal.h"

namespace zr {
namespace {

constexpr int kMaxPlanRows = 8192;
constexpr int kCachedPackEntries = 1024;  // 24 KB of shared memory per block

// Per row: valid prompt / response token counts and whether the mask has the
// supported shape (prompt left padded, response right padded).
__global__ void mask_rows_kernel(const uint8_t* __restrict__ mask, int L, int P,
                                 int32_t* __restrict__ row_plen, int32_t* __restrict__ row_rlen,
                                 int32_t* __restrict__ status) {
    const int b = blockIdx.x;
    int c1 = 0, f1 = P, l1 = -1, c2 = 0, f2 = L, l2 = P - 1;
    if (mask) {
        const uint8_t* m = mask + (int64_t)b * L;
        for (int i = threadIdx.x; i < L; i += blockDim.x) {
            if (m[i] != 0) {
                if (i < P) { ++c1; f1 = min(f1, i); l1 = max(l1, i); }
                else { ++c2; f2 = min(f2, i); l2 = max(l2, i); }
            }
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        c1 += __shfl_xor_sync(0xffffffffu, c1, o);
        c2 += __shfl_xor_sync(0xffffffffu, c2, o);
        f1 = min(f1, __shfl_xor_sync(0xffffffffu, f1, o));
        f2 = min(f2, __shfl_xor_sync(0xffffffffu, f2, o));
        l1 = max(l1, __shfl_xor_sync(0xffffffffu, l1, o));
        l2 = max(l2, __shfl_xor_sync(0xffffffffu, l2, o));
    }
    __shared__ int red[6][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        red[0][warp] = c1; red[1][warp] = c2; red[2][warp] = f1;
        red[3][warp] = f2; red[4][warp] = l1; red[5][warp] = l2;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!mask) {
            row_plen[b] = P;
            row_rlen[b] = L - P;
            return;
        }
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
            red[0][0] += red[0][w]; red[1][0] += red[1][w];
            red[2][0] = min(red[2][0], red[2][w]); red[3][0] = min(red[3][0], red[3][w]);
            red[4][0] = max(red[4][0], red[4][w]); red[5][0] = max(red[5][0], red[5][w]);
        }
        c1 = red[0][0]; c2 = red[1][0];
        f1 = red[2][0]; f2 = red[3][0]; l1 = red[4][0]; l2 = red[5][0];
        const bool prompt_ok = (c1 == 0) || (l1 == P - 1 && f1 == P - c1);
        const bool resp_ok = (c2 == 0) || (f2 == P && l2 == P + c2 - 1);
        row_plen[b] = c1;
        row_rlen[b] = c2;
        if (!(prompt_ok && resp_ok)) atomicExch(&status[kStatusMask], (int)ZR_ERR_INVALID_ARG);
    }
}

__device__ int block_exclusive_scan_i32(int* data, int n) {
    __shared__ int warp_tot[32];
    const int nthr = blockDim.x;
    const int per = (n + nthr - 1) / nthr;
    const int lo = min(threadIdx.x * per, n), hi = min(lo + per, n);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += data[i];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = nthr >> 5;
    int x = sum;
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nwarp ? warp_tot[lane] : 0;
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_tot[lane] = w;
    }
    __syncthreads();
    int run = x - sum + (warp > 0 ? warp_tot[warp - 1] : 0);
    const int total = warp_tot[nwarp - 1];
    for (int i = lo; i < hi; ++i) {
        int v = data[i];
        data[i] = run;
        run += v;
    }
    __syncthreads();
    return total;
}

struct PlanArgs {
    const int32_t* gptr; const int32_t* gmem; const int32_t* gof; const int32_t* ng;
    zr_recon_info info;
    int R;
};

__device__ __forceinline__ void put_seg(int64_t* segs, int i, int64_t src, int64_t dst, int64_t n) {
    segs[3 * i + 0] = src;
    segs[3 * i + 1] = dst;
    segs[3 * i + 2] = n;
}

// Slot offsets, T and the three segment tables.  One block.
__global__ void pack_plan_kernel(PlanArgs a) {
    extern __shared__ int smem[];
    const zr_recon_info& in = a.info;
    const int B = in.B, L = in.L, P = in.P, R = a.R;
    const bool unpad = in.use_unpad != 0;
    int* s_pslot = smem;        // [B] prompt slot rows per group (0 past G)
    int* s_rslot = smem + B;    // [B] response slot rows in CSR member order
    const int G = a.ng[0];
    const bool bad_mask = in.status[kStatusMask] != 0;
    for (int i = threadIdx.x; i < B; i += blockDim.x) {
        int ps = 0;
        if (i < G) {
            const int rep = a.gmem[a.gptr[i]];
            ps = unpad ? in.row_prompt_len[rep] : P;
        }
        s_pslot[i] = ps;
        const int b = a.gmem[i];
        s_rslot[i] = unpad ? in.resp_len[b] : R;
    }
    __syncthreads();
    // keep the slot sizes (the scans overwrite the arrays)
    for (int i = threadIdx.x; i < B; i += blockDim.x) {
        if (i < G) in.prompt_slot[i] = s_pslot[i];
        in.resp_slot[a.gmem[i]] = s_rslot[i];
    }
    __syncthreads();
    const int tot_p = block_exclusive_scan_i32(s_pslot, B);
    const int tot_r = block_exclusive_scan_i32(s_rslot, B);
    const int64_t T = bad_mask ? 0 : (int64_t)tot_p + tot_r;
    const int64_t cap = in.T_cap;
    for (int g = threadIdx.x; g < B; g += blockDim.x) {
        if (g < G) {
            const int rep = a.gmem[a.gptr[g]];
            const int ps = in.prompt_slot[g];
            const int pl = in.row_prompt_len[rep];
            const int off = s_pslot[g] + s_rslot[a.gptr[g]];
            in.prompt_off[g] = off;
            in.prompt_len[g] = pl;
            const int64_t n = bad_mask ? 0 : ps;
            const int64_t n_fit = max((int64_t)0, min(n, cap - off));
            put_seg(in.pack_segs, g, (int64_t)rep * L + (P - ps), off, n_fit);
            put_seg(in.pad_segs, g, -1, off, bad_mask ? 0 : max((int64_t)0, min((int64_t)(ps - pl), cap - off)));
        } else {
            put_seg(in.pack_segs, g, -1, 0, 0);
            put_seg(in.pad_segs, g, -1, 0, 0);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < B; i += blockDim.x) {
        const int b = a.gmem[i];
        const int g = a.gof[b];
        const int off = s_pslot[g] + in.prompt_slot[g] + s_rslot[i];
        const int rs = in.resp_slot[b];
        const int rl = in.resp_len[b];
        in.resp_off[b] = off;
        in.group_of[b] = g;
        const int64_t n = bad_mask ? 0 : rs;
        put_seg(in.pack_segs, B + b, (int64_t)b * L + P, off, max((int64_t)0, min(n, cap - off)));
        const int64_t pad_lo = (int64_t)off + rl;
        put_seg(in.pad_segs, B + b, -1, pad_lo,
                bad_mask ? 0 : max((int64_t)0, min((int64_t)(rs - rl), cap - pad_lo)));
        // reconstruction of row b: prompt, prompt pad, response, response pad
        const int po = in.prompt_off[g];
        const int ps = in.prompt_slot[g];
        const bool ok = !bad_mask && (T <= cap);
        put_seg(in.recon_segs, 4 * b + 0, po, (int64_t)b * L + (P - ps), ok ? ps : 0);
        put_seg(in.recon_segs, 4 * b + 1, -1, (int64_t)b * L, ok ? P - ps : P);
        put_seg(in.recon_segs, 4 * b + 2, off, (int64_t)b * L + P, ok ? rs : 0);
        put_seg(in.recon_segs, 4 * b + 3, -1, (int64_t)b * L + P + (ok ? rs : 0), ok ? R - rs : R);
    }
    __syncthreads();
    // the pack segments in packed-row order: group g's prompt (entry
    // group_ptr[g] + g), then each member's response (entry q + g + 1 for CSR
    // position q); entries past G + B are empty and sort last
    for (int q = threadIdx.x; q < B; q += blockDim.x) {
        const int b = a.gmem[q];
        const int g = a.gof[b];
        const int64_t* r = in.pack_segs + 3 * (int64_t)(B + b);
        put_seg(in.pack_order, q + g + 1, r[0], r[1], r[2]);
        if (a.gptr[g] == q) {
            const int64_t* pr = in.pack_segs + 3 * (int64_t)g;
            put_seg(in.pack_order, q + g, pr[0], pr[1], pr[2]);
        }
        if (q >= G) put_seg(in.pack_order, B + q, -1, INT64_MAX, 0);
    }
    for (int i = threadIdx.x; i <= B; i += blockDim.x) in.group_ptr[i] = a.gptr[i];
    for (int i = threadIdx.x; i < B; i += blockDim.x) in.members[i] = a.gmem[i];
    if (threadIdx.x == 0) {
        in.num_groups[0] = G;
        in.total_tokens[0] = (int)T;
        if (T > cap) atomicExch(&in.status[kStatusCapacity], (int)ZR_ERR_CAPACITY);
    }
}

// Copies (src row >= 0) or zero-fills (src row < 0) every segment of a table.
// blockIdx.y selects the segment, blockIdx.x strides over its bytes.
template <bool kStreamStores>
__global__ void __launch_bounds__(256) segment_copy_kernel(const char* __restrict__ src,
                                                           char* __restrict__ dst,
                                                           const int64_t* __restrict__ segs,
                                                           int64_t row_bytes) {
    const int s = blockIdx.y;
    const int64_t src_row = segs[3 * s + 0];
    const int64_t dst_row = segs[3 * s + 1];
    const int64_t nrows = segs[3 * s + 2];
    if (nrows <= 0) return;
    const int64_t bytes = nrows * row_bytes;
    char* d = dst + dst_row * row_bytes;
    const char* sp = (src_row >= 0) ? src + src_row * row_bytes : nullptr;
    const uintptr_t align = (uintptr_t)d | (uintptr_t)sp | (uintptr_t)bytes;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
    if ((align & 15) == 0) {
        const int64_t nv = bytes >> 4;
        int4* d4 = reinterpret_cast<int4*>(d);
        const int4* s4 = reinterpret_cast<const int4*>(sp);
        constexpr int U = 4;
        int64_t i = tid;
        for (; i + (U - 1) * nthr < nv; i += U * nthr) {
            int4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) v[u] = sp ? __ldg(s4 + i + u * nthr) : make_int4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (kStreamStores) __stcs(d4 + i + u * nthr, v[u]);
                else d4[i + u * nthr] = v[u];
            }
        }
        for (; i < nv; i += nthr) {
            int4 v = sp ? __ldg(s4 + i) : make_int4(0, 0, 0, 0);
            if (kStreamStores) __stcs(d4 + i, v);
            else d4[i] = v;
        }
    } else if ((align & 7) == 0) {
        const int64_t nv = bytes >> 3;
        long long* d8 = reinterpret_cast<long long*>(d);
        const long long* s8 = reinterpret_cast<const long long*>(sp);
        for (int64_t i = tid; i < nv; i += nthr) d8[i] = sp ? __ldg(s8 + i) : 0ll;
    } else {
        for (int64_t i = tid; i < bytes; i += nthr) d[i] = sp ? sp[i] : (char)0;
    }
}

// Copies (sp != nullptr) or zero-fills `bytes` contiguous bytes with every
// thread of the block.  Full passes issue eight 16-byte loads per thread before
// the matching stores; the tail goes one vector at a time.
__device__ __forceinline__ int4 load16(const int4* p) { return __ldg(p); }

template <bool kStreamStores>
__device__ __forceinline__ void store16(int4* p, int4 v) {
    if (kStreamStores) __stcs(p, v);
    else *p = v;
}

template <bool kStreamStores>
__device__ __forceinline__ void block_copy(const char* __restrict__ sp, char* __restrict__ d,
                                           int64_t bytes) {
    const uintptr_t align = (uintptr_t)d | (uintptr_t)sp | (uintptr_t)bytes;
    const int nthr = blockDim.x;
    if ((align & 15) == 0) {
        const int64_t nv = bytes >> 4;
        int4* d4 = reinterpret_cast<int4*>(d);
        const int4* s4 = reinterpret_cast<const int4*>(sp);
        constexpr int U = 8;
        int64_t i = threadIdx.x;
        if (sp) {
            for (; i + (int64_t)(U - 1) * nthr < nv; i += (int64_t)U * nthr) {
                int4 v[U];
#pragma unroll
                for (int u = 0; u < U; ++u) v[u] = load16(s4 + i + (int64_t)u * nthr);
#pragma unroll
                for (int u = 0; u < U; ++u) store16<kStreamStores>(d4 + i + (int64_t)u * nthr, v[u]);
            }
            for (; i < nv; i += nthr) store16<kStreamStores>(d4 + i, load16(s4 + i));
        } else {
            const int4 z = make_int4(0, 0, 0, 0);
            for (; i < nv; i += nthr) store16<kStreamStores>(d4 + i, z);
        }
    } else if ((align & 7) == 0) {
        const int64_t nv = bytes >> 3;
        long long* d8 = reinterpret_cast<long long*>(d);
        const long long* s8 = reinterpret_cast<const long long*>(sp);
        for (int64_t i = threadIdx.x; i < nv; i += nthr) d8[i] = sp ? __ldg(s8 + i) : 0ll;
    } else {
        for (int64_t i = threadIdx.x; i < bytes; i += nthr) d[i] = sp ? sp[i] : (char)0;
    }
}

// Packing, output-stationary: the packed rows [0, T) are cut into work items
// of chunk_rows rows; an item finds the pack segment holding its first row by
// binary search over the segments sorted by packed row, then copies the rows
// of every segment it overlaps.  Persistent blocks stride over the items.
// With kCached the block first copies the (small) segment table into shared
// memory, so the searches cost no global round trips.
template <bool kCached>
__global__ void __launch_bounds__(256) pack_rows_kernel(const char* __restrict__ src,
                                                        char* __restrict__ dst,
                                                        const int64_t* __restrict__ order,
                                                        int n_entries,
                                                        const int32_t* __restrict__ total_tokens,
                                                        int64_t T_cap, int chunk_rows,
                                                        int64_t row_bytes, int64_t src_rows,
                                                        int32_t* __restrict__ status) {
    extern __shared__ int64_t s_order[];
    const int64_t T = min((int64_t)total_tokens[0], T_cap);
    const int64_t* ord = order;
    if (kCached) {
        for (int i = threadIdx.x; i < 3 * n_entries; i += blockDim.x) s_order[i] = order[i];
        __syncthreads();
        ord = s_order;
    }
    const int64_t items = (T + chunk_rows - 1) / chunk_rows;
    for (int64_t k = blockIdx.x; k < items; k += gridDim.x) {
        const int64_t r0 = k * chunk_rows;
        const int64_t r1 = min(T, r0 + chunk_rows);
        // largest j with ord[j].dst <= r0 (entry 0 starts at packed row 0)
        int lo = 0, hi = n_entries - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (ord[3 * mid + 1] <= r0) lo = mid;
            else hi = mid - 1;
        }
        for (int j = lo; j < n_entries; ++j) {
            const int64_t s0 = ord[3 * j + 0];
            const int64_t d0 = ord[3 * j + 1];
            const int64_t n = ord[3 * j + 2];
            if (d0 >= r1) break;
            const int64_t a = max(d0, r0), e = min(d0 + n, r1);
            if (a < e && s0 >= 0 && ZR_BOUNDS(s0 + (e - d0) <= src_rows && e <= T_cap, status, 1))
                block_copy<false>(src + (s0 + (a - d0)) * row_bytes, dst + a * row_bytes,
                                  (e - a) * row_bytes);
        }
    }
}

// Reconstruction adjoint, output-stationary over the packed rows like the pack:
// packed row x of pack segment (s0, d0, n) receives the sum, over the
// segment's members b, of grad_out row b*L + (s0 mod L) + (x - d0).  A
// response segment (s0 mod L == P) has the one member s0 / L; a prompt
// segment (s0 mod L < P) has every member of the group of its representative
// s0 / L.  Sums run in fp32 over the members in group order; elements are bf16
// or fp32 (ElemT), 16-byte vectors when rows allow it.
__device__ __forceinline__ uint32_t pack_rne_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ void acc16(float (&a)[8], uint4 v, __nv_bfloat16) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        a[2 * i] += __uint_as_float(w[i] << 16);
        a[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void acc16(float (&a)[8], uint4 v, float) {
    a[0] += __uint_as_float(v.x);
    a[1] += __uint_as_float(v.y);
    a[2] += __uint_as_float(v.z);
    a[3] += __uint_as_float(v.w);
}
__device__ __forceinline__ uint4 out16(const float (&a)[8], __nv_bfloat16) {
    uint4 r;
    r.x = pack_rne_bf16x2(a[0], a[1]);
    r.y = pack_rne_bf16x2(a[2], a[3]);
    r.z = pack_rne_bf16x2(a[4], a[5]);
    r.w = pack_rne_bf16x2(a[6], a[7]);
    return r;
}
__device__ __forceinline__ uint4 out16(const float (&a)[8], float) {
    return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                      __float_as_uint(a[3]));
}
__device__ __forceinline__ float elem_to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float elem_to_f(float x) { return x; }
__device__ __forceinline__ void f_to_elem(float v, __nv_bfloat16* p) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ void f_to_elem(float v, float* p) { *p = v; }

template <typename ElemT, bool kCached>
__global__ void __launch_bounds__(256) reconstruct_backward_kernel(const ElemT* __restrict__ gout,
                                                                   ElemT* __restrict__ gpacked,
                                                                   zr_recon_info info, int n_entries,
                                                                   int chunk_rows, int64_t W) {
    extern __shared__ int64_t s_order[];
    const int64_t T = min((int64_t)info.total_tokens[0], info.T_cap);
    const int64_t* ord = info.pack_order;
    if (kCached) {
        for (int i = threadIdx.x; i < 3 * n_entries; i += blockDim.x) s_order[i] = info.pack_order[i];
        __syncthreads();
        ord = s_order;
    }
    const int L = info.L;
    constexpr int kPerVec = 16 / sizeof(ElemT);
    const bool vec = ((W * (int64_t)sizeof(ElemT)) & 15) == 0 && (((uintptr_t)gout | (uintptr_t)gpacked) & 15) == 0;
    const int64_t items = (T + chunk_rows - 1) / chunk_rows;
    for (int64_t k = blockIdx.x; k < items; k += gridDim.x) {
        const int64_t r0 = k * chunk_rows;
        const int64_t r1 = min(T, r0 + chunk_rows);
        int lo = 0, hi = n_entries - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (ord[3 * mid + 1] <= r0) lo = mid;
            else hi = mid - 1;
        }
        for (int j = lo; j < n_entries; ++j) {
            const int64_t s0 = ord[3 * j + 0];
            const int64_t d0 = ord[3 * j + 1];
            const int64_t n = ord[3 * j + 2];
            if (d0 >= r1) break;
            const int64_t a = max(d0, r0), e = min(d0 + n, r1);
            if (a >= e || s0 < 0) continue;
            if (!ZR_BOUNDS(s0 + (e - d0) <= (int64_t)info.B * L && e <= info.T_cap, info.status, 3)) continue;
            const int rep = (int)(s0 / L);
            const int64_t col = s0 - (int64_t)rep * L + (a - d0);  // row offset inside each member's row
            int mb = 0, me = 1;
            const bool prompt = (s0 - (int64_t)rep * L) < info.P;
            if (prompt) {
                const int g = info.group_of[rep];
                mb = info.group_ptr[g];
                me = info.group_ptr[g + 1];
                if (!ZR_BOUNDS(mb >= 0 && mb < me && me <= info.B, info.status, 4)) continue;
            }
            const int64_t nel = (e - a) * W;
            ElemT* dst = gpacked + a * W;
            if (vec) {
                // two vectors per thread, members four at a time: up to eight
                // independent 16-byte loads in flight per thread
                const int64_t nv = nel / kPerVec;
                const int64_t stride = blockDim.x;
                for (int64_t v = threadIdx.x; v < nv; v += 2 * stride) {
                    const bool two = v + stride < nv;
                    float acc0[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                    float acc1[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                    int m = mb;
                    for (; m + 4 <= me; m += 4) {
                        uint4 x0[4], x1[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int b = prompt ? info.members[m + q] : rep;
                            const uint4* src = reinterpret_cast<const uint4*>(gout + ((int64_t)b * L + col) * W);
                            x0[q] = __ldg(src + v);
                            x1[q] = two ? __ldg(src + v + stride) : make_uint4(0u, 0u, 0u, 0u);
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            acc16(acc0, x0[q], ElemT());
                            acc16(acc1, x1[q], ElemT());
                        }
                    }
                    for (; m < me; ++m) {
                        const int b = prompt ? info.members[m] : rep;
                        const uint4* src = reinterpret_cast<const uint4*>(gout + ((int64_t)b * L + col) * W);
                        acc16(acc0, __ldg(src + v), ElemT());
                        if (two) acc16(acc1, __ldg(src + v + stride), ElemT());
                    }
                    reinterpret_cast<uint4*>(dst)[v] = out16(acc0, ElemT());
                    if (two) reinterpret_cast<uint4*>(dst)[v + stride] = out16(acc1, ElemT());
                }
            } else {
                for (int64_t v = threadIdx.x; v < nel; v += blockDim.x) {
                    float acc = 0.f;
                    for (int m = mb; m < me; ++m) {
                        const int b = prompt ? info.members[m] : rep;
                        acc += elem_to_f(gout[((int64_t)b * L + col) * W + v]);
                    }
                    f_to_elem(acc, dst + v);
                }
            }
        }
    }
}

// Reconstruction, output-stationary: every output row range is written once.
// The work items are (row b, chunk c of chunk_rows rows of b) and are ordered
// group by group, chunk by chunk, member by member, so the members of a group
// that copy the same chunk of the shared prompt run side by side and all but
// the first find it in L2: the packed prompt is read from DRAM about once.
// Each item intersects its row range with the four reconstruction segments of
// row b (prompt pad, prompt, response, response pad) and copies or zero-fills
// the overlaps.  Persistent blocks stride over the items.
//
// With kPackAdjoint the same walk computes the adjoint of the pack: source
// position (b, p) receives the gradient of the packed row that was read from
// it.  The pack reads a group's prompt from its representative (the first
// member) only, so the prompt segment of every other member is zero-filled;
// everything else is the reconstruction's copy.
template <bool kPackAdjoint>
__global__ void __launch_bounds__(256) reconstruct_rows_kernel(const char* __restrict__ packed,
                                                               char* __restrict__ out,
                                                               zr_recon_info info, int chunk_rows,
                                                               int64_t nchunks, int64_t row_bytes) {
    const int L = info.L;
    const int64_t items = (int64_t)info.B * nchunks;
    for (int64_t k = blockIdx.x; k < items; k += gridDim.x) {
        const int q = (int)(k / nchunks);                // member position (CSR order)
        const int g = info.group_of[info.members[q]];
        const int base = info.group_ptr[g];
        const int n = info.group_ptr[g + 1] - base;
        if (n <= 0 || !ZR_BOUNDS(base >= 0 && base + n <= info.B, info.status, 5)) continue;
        const int64_t local = k - (int64_t)base * nchunks;
        const int64_t c = local / n;
        const int b = info.members[base + (int)(local % n)];
        const bool rep = b == info.members[base];
        const int64_t r0 = c * chunk_rows;
        const int64_t r1 = min((int64_t)L, r0 + chunk_rows);
        const int64_t row0 = (int64_t)b * L;
        for (int sgi = 0; sgi < 4; ++sgi) {
            const int64_t* seg = info.recon_segs + 3 * (4 * (int64_t)b + sgi);
            const int64_t src = (kPackAdjoint && sgi == 0 && !rep) ? -1 : seg[0];
            const int64_t lo = seg[1] - row0, nrows = seg[2];
            const int64_t a = max(lo, r0), e = min(lo + nrows, r1);
            if (a >= e || !ZR_BOUNDS(src < 0 || src + (e - lo) <= info.T_cap, info.status, 2)) continue;
            block_copy<true>(src >= 0 ? packed + (src + (a - lo)) * row_bytes : nullptr,
                             out + (row0 + a) * row_bytes, (e - a) * row_bytes);
        }
    }
}

// The gradient of reconstruct(pack(x)) with respect to x in one pass, for a
// tensor that is packed, carried unchanged and reconstructed (the adjoint of
// the reconstruction followed by the adjoint of the pack, without the packed
// intermediate).  Output-stationary over [B, L] like the reconstruction: the
// representative of a group receives, at each prompt position the pack read,
// the fp32 sum over the group's members (in group order, rounded once) of
// grad_out there; the prompt rows of the other members are zero; every row's
// packed response positions pass their own gradient through; positions the
// pack dropped or never read are zero.
template <typename ElemT>
__global__ void __launch_bounds__(256) reconstruct_pack_backward_kernel(const ElemT* __restrict__ gout,
                                                                        ElemT* __restrict__ gin,
                                                                        zr_recon_info info, int chunk_rows,
                                                                        int64_t nchunks, int64_t W) {
    const int L = info.L;
    const int64_t row_bytes = W * (int64_t)sizeof(ElemT);
    constexpr int kPerVec = 16 / sizeof(ElemT);
    const bool vec = (row_bytes & 15) == 0 && (((uintptr_t)gout | (uintptr_t)gin) & 15) == 0;
    const int64_t items = (int64_t)info.B * nchunks;
    for (int64_t k = blockIdx.x; k < items; k += gridDim.x) {
        const int q = (int)(k / nchunks);
        const int g = info.group_of[info.members[q]];
        const int base = info.group_ptr[g];
        const int n = info.group_ptr[g + 1] - base;
        if (n <= 0 || !ZR_BOUNDS(base >= 0 && base + n <= info.B, info.status, 6)) continue;
        const int64_t local = k - (int64_t)base * nchunks;
        const int64_t c = local / n;
        const int b = info.members[base + (int)(local % n)];
        const bool rep = b == info.members[base];
        const int64_t r0 = c * chunk_rows;
        const int64_t r1 = min((int64_t)L, r0 + chunk_rows);
        const int64_t row0 = (int64_t)b * L;
        for (int sgi = 0; sgi < 4; ++sgi) {
            const int64_t* seg = info.recon_segs + 3 * (4 * (int64_t)b + sgi);
            const int64_t lo = seg[1] - row0, nrows = seg[2];
            const int64_t a = max(lo, r0), e = min(lo + nrows, r1);
            if (a >= e) continue;
            char* dst = reinterpret_cast<char*>(gin + (row0 + a) * W);
            if (seg[0] < 0 || (sgi == 0 && !rep)) {  // pads, other members' prompts
                block_copy<false>(nullptr, dst, (e - a) * row_bytes);
                continue;
            }
            if (sgi == 2) {  // the row's own response rows
                block_copy<false>(reinterpret_cast<const char*>(gout + (row0 + a) * W), dst, (e - a) * row_bytes);
                continue;
            }
            // the representative's prompt rows: sum over the group's members
            const int64_t nel = (e - a) * W;
            ElemT* d = gin + (row0 + a) * W;
            if (vec) {
                const int64_t nv = nel / kPerVec;
                for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) {
                    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                    int m = base;
                    for (; m + 4 <= base + n; m += 4) {
                        uint4 x[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            x[u] = __ldg(reinterpret_cast<const uint4*>(gout + ((int64_t)info.members[m + u] * L + a) * W) + v);
#pragma unroll
                        for (int u = 0; u < 4; ++u) acc16(acc, x[u], ElemT());
                    }
                    for (; m < base + n; ++m)
                        acc16(acc, __ldg(reinterpret_cast<const uint4*>(gout + ((int64_t)info.members[m] * L + a) * W) + v),
                              ElemT());
                    reinterpret_cast<uint4*>(d)[v] = out16(acc, ElemT());
                }
            } else {
                for (int64_t v = threadIdx.x; v < nel; v += blockDim.x) {
                    float acc = 0.f;
                    for (int m = base; m < base + n; ++m)
                        acc += elem_to_f(gout[((int64_t)info.members[m] * L + a) * W + v]);
                    f_to_elem(acc, d + v);
                }
            }
        }
    }
}

// Batch statistics from the per-row valid prompt / response counts: one block.
__global__ void batch_stats_kernel(const int32_t* __restrict__ plen, const int32_t* __restrict__ rlen, int B,
                                   int L, zr_batch_stats* __restrict__ out) {
    __shared__ long long s_sum[2][32];
    __shared__ int s_min[2][32], s_max[2][32], s_cnt[32];
    long long sp = 0, sr = 0;
    int pmin = INT_MAX, pmax = 0, rmin = INT_MAX, rmax = 0, cnt = 0;
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        const int p = plen[b], r = rlen[b];
        sp += p;
        pmin = min(pmin, p);
        pmax = max(pmax, p);
        if (r > 0) {
            sr += r;
            rmin = min(rmin, r);
            rmax = max(rmax, r);
            ++cnt;
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        sp += __shfl_xor_sync(0xffffffffu, sp, o);
        sr += __shfl_xor_sync(0xffffffffu, sr, o);
        pmin = min(pmin, __shfl_xor_sync(0xffffffffu, pmin, o));
        pmax = max(pmax, __shfl_xor_sync(0xffffffffu, pmax, o));
        rmin = min(rmin, __shfl_xor_sync(0xffffffffu, rmin, o));
        rmax = max(rmax, __shfl_xor_sync(0xffffffffu, rmax, o));
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (lane == 0) {
        s_sum[0][warp] = sp; s_sum[1][warp] = sr;
        s_min[0][warp] = pmin; s_max[0][warp] = pmax;
        s_min[1][warp] = rmin; s_max[1][warp] = rmax;
        s_cnt[warp] = cnt;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < nw; ++w) {
            s_sum[0][0] += s_sum[0][w]; s_sum[1][0] += s_sum[1][w];
            s_min[0][0] = min(s_min[0][0], s_min[0][w]); s_max[0][0] = max(s_max[0][0], s_max[0][w]);
            s_min[1][0] = min(s_min[1][0], s_min[1][w]); s_max[1][0] = max(s_max[1][0], s_max[1][w]);
            s_cnt[0] += s_cnt[w];
        }
        const long long total = (long long)B * L;
        const int nr = s_cnt[0];
        out->rows = B;
        out->responses = nr;
        out->non_pad_tokens = s_sum[0][0] + s_sum[1][0];
        out->total_positions = total;
        out->prompt_len_min = B > 0 ? s_min[0][0] : 0;
        out->prompt_len_max = s_max[0][0];
        out->resp_len_min = nr > 0 ? s_min[1][0] : 0;
        out->resp_len_max = nr > 0 ? s_max[1][0] : 0;
        out->prompt_len_mean = B > 0 ? (double)s_sum[0][0] / B : 0.0;
        out->resp_len_mean = nr > 0 ? (double)s_sum[1][0] / nr : 0.0;
        out->non_pad_fraction = total > 0 ? (double)(s_sum[0][0] + s_sum[1][0]) / (double)total : 0.0;
    }
}

int blocks_for(int64_t max_seg_bytes) {
    // one block streams 16 KB per pass; cap the x extent
    int64_t x = (max_seg_bytes + 16383) / 16384;
    if (x < 1) x = 1;
    if (x > 256) x = 256;
    return (int)x;
}

}  // namespace

zr_status launch_pack_plan(const zr_groups& g, const uint8_t* mask, const zr_recon_info& info,
                           cudaStream_t s) {
    const int B = info.B;
    if (B > kMaxPlanRows) return set_error(ZR_ERR_UNSUPPORTED, "B=%d exceeds %d rows", B, kMaxPlanRows);
    ZR_CUDA_TRY(cudaMemsetAsync(info.status, 0, 4 * sizeof(int32_t), s));
    mask_rows_kernel<<<B, 256, 0, s>>>(mask, info.L, info.P, info.row_prompt_len, info.resp_len,
                                       info.status);
    ZR_LAUNCH_CHECK("mask_rows_kernel");
    PlanArgs a;
    a.gptr = g.group_ptr; a.gmem = g.members; a.gof = g.group_of; a.ng = g.num_groups;
    a.info = info;
    a.R = info.L - info.P;
    const int smem = 2 * B * (int)sizeof(int);
    ZR_CUDA_TRY(cudaFuncSetAttribute(pack_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     2 * kMaxPlanRows * (int)sizeof(int)));
    pack_plan_kernel<<<1, 1024, smem, s>>>(a);
    ZR_LAUNCH_CHECK("pack_plan_kernel");
    return ZR_OK;
}

zr_status launch_pack_gather(const zr_recon_info& info, const void* src, int64_t row_bytes,
                             void* dst, cudaStream_t s) {
    // work items of 4-32 KB: about one pass of block_copy each, and enough
    // items to occupy every SM when the tensor is small
    const int64_t blocks = (int64_t)num_sms() * 8;
    const int64_t item_bytes = std::min<int64_t>(32768, std::max<int64_t>(4096, info.T_cap * row_bytes / blocks));
    const int chunk_rows = (int)std::max<int64_t>(1, std::min<int64_t>(info.T_cap, item_bytes / row_bytes));
    const int64_t items = (info.T_cap + chunk_rows - 1) / chunk_rows;
    const int grid = (int)std::min<int64_t>(items, blocks);
    const int n_entries = 2 * info.B;
    KernelTimer timer("pack_gather", s);
    if (n_entries <= kCachedPackEntries) {
        pack_rows_kernel<true><<<grid, 256, (size_t)n_entries * 24, s>>>(
            static_cast<const char*>(src), static_cast<char*>(dst), info.pack_order, n_entries,
            info.total_tokens, info.T_cap, chunk_rows, row_bytes, (int64_t)info.B * info.L, info.status);
    } else {
        pack_rows_kernel<false><<<grid, 256, 0, s>>>(
            static_cast<const char*>(src), static_cast<char*>(dst), info.pack_order, n_entries,
            info.total_tokens, info.T_cap, chunk_rows, row_bytes, (int64_t)info.B * info.L, info.status);
    }
    ZR_LAUNCH_CHECK("pack_rows_kernel");
    return ZR_OK;
}

zr_status launch_reconstruct(const zr_recon_info& info, const void* packed, int64_t row_bytes,
                             void* out, cudaStream_t s) {
    // about 32 KB of output per work item: one pass of block_copy
    const int chunk_rows = (int)std::max<int64_t>(1, std::min<int64_t>(info.L, 32768 / row_bytes));
    const int64_t nchunks = (info.L + chunk_rows - 1) / chunk_rows;
    const int64_t items = (int64_t)info.B * nchunks;
    const int grid = (int)std::min<int64_t>(items, (int64_t)num_sms() * 8);
    KernelTimer timer("reconstruct", s);
    reconstruct_rows_kernel<false><<<grid, 256, 0, s>>>(static_cast<const char*>(packed),
                                                        static_cast<char*>(out), info, chunk_rows, nchunks,
                                                        row_bytes);
    ZR_LAUNCH_CHECK("reconstruct_rows_kernel");
    return ZR_OK;
}

zr_status launch_pack_backward(const zr_recon_info& info, const void* grad_packed, int64_t row_bytes,
                               void* grad_src, cudaStream_t s) {
    const int chunk_rows = (int)std::max<int64_t>(1, std::min<int64_t>(info.L, 32768 / row_bytes));
    const int64_t nchunks = (info.L + chunk_rows - 1) / chunk_rows;
    const int64_t items = (int64_t)info.B * nchunks;
    const int grid = (int)std::min<int64_t>(items, (int64_t)num_sms() * 8);
    KernelTimer timer("pack_backward", s);
    reconstruct_rows_kernel<true><<<grid, 256, 0, s>>>(static_cast<const char*>(grad_packed),
                                                       static_cast<char*>(grad_src), info, chunk_rows, nchunks,
                                                       row_bytes);
    ZR_LAUNCH_CHECK("reconstruct_rows_kernel(pack adjoint)");
    return ZR_OK;
}

zr_status launch_reconstruct_pack_backward(const zr_recon_info& info, const void* grad_out, int64_t W,
                                           zr_dtype dtype, void* grad_in, cudaStream_t s) {
    const int64_t row_bytes = W * (dtype == ZR_F32 ? 4 : 2);
    const int chunk_rows = (int)std::max<int64_t>(1, std::min<int64_t>(info.L, 32768 / row_bytes));
    const int64_t nchunks = (info.L + chunk_rows - 1) / chunk_rows;
    const int64_t items = (int64_t)info.B * nchunks;
    const int grid = (int)std::min<int64_t>(items, (int64_t)num_sms() * 8);
    KernelTimer timer("reconstruct_pack_backward", s);
    if (dtype == ZR_F32)
        reconstruct_pack_backward_kernel<float><<<grid, 256, 0, s>>>(
            static_cast<const float*>(grad_out), static_cast<float*>(grad_in), info, chunk_rows, nchunks, W);
    else
        reconstruct_pack_backward_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(grad_out), static_cast<__nv_bfloat16*>(grad_in), info, chunk_rows,
            nchunks, W);
    ZR_LAUNCH_CHECK("reconstruct_pack_backward_kernel");
    return ZR_OK;
}

zr_status launch_reconstruct_backward(const zr_recon_info& info, const void* grad_out, int64_t W,
                                      zr_dtype dtype, void* grad_packed, cudaStream_t s) {
    const int64_t row_bytes = W * (dtype == ZR_F32 ? 4 : 2);
    const int64_t blocks = (int64_t)num_sms() * 8;
    const int64_t item_bytes = std::min<int64_t>(32768, std::max<int64_t>(4096, info.T_cap * row_bytes / blocks));
    const int chunk_rows = (int)std::max<int64_t>(1, std::min<int64_t>(info.T_cap, item_bytes / row_bytes));
    const int64_t items = (info.T_cap + chunk_rows - 1) / chunk_rows;
    const int grid = (int)std::min<int64_t>(items, blocks);
    const int n_entries = 2 * info.B;
    const bool cached = n_entries <= kCachedPackEntries;
    const size_t smem = cached ? (size_t)n_entries * 24 : 0;
    KernelTimer timer("reconstruct_backward", s);
    if (dtype == ZR_F32) {
        const float* g = static_cast<const float*>(grad_out);
        float* o = static_cast<float*>(grad_packed);
        if (cached) reconstruct_backward_kernel<float, true><<<grid, 256, smem, s>>>(g, o, info, n_entries, chunk_rows, W);
        else reconstruct_backward_kernel<float, false><<<grid, 256, 0, s>>>(g, o, info, n_entries, chunk_rows, W);
    } else {
        const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(grad_out);
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(grad_packed);
        if (cached)
            reconstruct_backward_kernel<__nv_bfloat16, true><<<grid, 256, smem, s>>>(g, o, info, n_entries, chunk_rows, W);
        else
            reconstruct_backward_kernel<__nv_bfloat16, false><<<grid, 256, 0, s>>>(g, o, info, n_entries, chunk_rows, W);
    }
    ZR_LAUNCH_CHECK("reconstruct_backward_kernel");
    return ZR_OK;
}

zr_status launch_batch_stats(const uint8_t* mask, int B, int L, int P, int32_t* plen, int32_t* rlen,
                             int32_t* status, zr_batch_stats* dev_out, cudaStream_t s) {
    mask_rows_kernel<<<B, 256, 0, s>>>(mask, L, P, plen, rlen, status);
    ZR_LAUNCH_CHECK("mask_rows_kernel");
    batch_stats_kernel<<<1, 1024, 0, s>>>(plen, rlen, B, L, dev_out);
    ZR_LAUNCH_CHECK("batch_stats_kernel");
    return ZR_OK;
}

zr_status launch_zero_pad_rows(const zr_recon_info& info, void* packed, int64_t row_bytes,
                               cudaStream_t s) {
    if (info.use_unpad) return ZR_OK;  // no pad rows in the unpadded layout
    const int64_t max_rows = info.P > info.L - info.P ? info.P : info.L - info.P;
    dim3 grid(blocks_for(max_rows * row_bytes), 2 * info.B);
    segment_copy_kernel<false><<<grid, 256, 0, s>>>(nullptr, static_cast<char*>(packed),
                                                    info.pad_segs, row_bytes);
    ZR_LAUNCH_CHECK("segment_copy_kernel(pad)");
    return ZR_OK;
}

}  // namespace zr
