// Split attention backward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// "How Prompt Deduplication Works", "Correctness & Gradients": gradients flow
// through the deduplicated attention; a prompt key's dK and dV collect the
// contributions of the prompt's own queries and of every response of its
// group.  The probabilities are recomputed from the forward's log-sum-exp:
// P = 2^(S * scale * log2(e) - LSE * log2(e)), dS = P * (dP - Delta) with
// Delta = rowsum(dO * O), dV = P^T dO, dK = scale * dS^T Q, dQ = scale * dS K.
// Each of the five GEMMs (S, dP, dV, dK, dQ) runs once per attended block.
//
// Three launches:
//   attn_bwd_prep_kernel     (-LSE * log2(e), Delta) pairs per (head, row),
//                            head-major, and zeroes the fp32 dQ accumulator
//   attn_bwd_tc_kernel       key-tile-major: per work unit (key tile, key/value
//                            head) the K and V tiles stay in shared memory while
//                            the query blocks that see them (all query heads of
//                            the group) stream through a TMA ring of 64-query
//                            halves (with the half's block descriptor and its
//                            -LSE/Delta, staged by the producer warp); per half,
//                            S^T = K Q^T and dP^T = V dO^T go to TMEM, the
//                            softmax warps write P^T and dS^T back
//                            to TMEM (bf16) and dS to shared memory, then
//                            dV += P^T dO, dK += dS^T Q (A operands from TMEM)
//                            and dQ^T = K^T dS^T (a per-half partial) run on the
//                            tensor cores; the softmax warps add each dQ^T
//                            partial into the fp32 accumulator (16-byte
//                            red.global.add.v4 into groups of four queries)
//   attn_dq_convert_kernel   dQ = scale * accumulator, rounded to bf16
// The query blocks that see a prompt key tile are the prompt's own blocks
// from the diagonal on (causal) and every block of every response of the
// group; a response key tile is seen by its own response's blocks from the
// diagonal on.  dQ sums over key tiles processed by different CTAs, so its
// fp32 accumulation order (and its last bits) can differ from run to run;
// dK and dV are accumulated in a fixed order.
//
// Every mbarrier wait is bounded (see zr_attn_tc.cu).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "zr_internal.h"
#include "zr_sm100.cuh"
#include "zr_tc_common.cuh"

namespace zr {
namespace {

using namespace sm100;
using namespace tc;


// st.shared.v4 without a compiler memory clobber: the proxy fence that
// follows these stores orders them (both are volatile asm)
__device__ __forceinline__ void st_shared_v4_nc(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d));
}

// 3-D tiled TMA load (x innermost)
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void st_shared_v2(uint32_t addr, float a, float b) {
    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}

// fire-and-forget fp32 add in global memory (performed at L2)
__device__ __forceinline__ void red_add_f32(float* addr, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}
// the same at a compile-time byte offset from `base` (no address arithmetic)
template <int kOffBytes>
__device__ __forceinline__ void red_add_f32_at(float* base, float v) {
    asm volatile("red.global.add.f32 [%0+%2], %1;" ::"l"(base), "f"(v), "n"(kOffBytes) : "memory");
}
template <int kOffBytes>
__device__ __forceinline__ void red_add_v2_at(float* base, uint32_t a, uint32_t b) {
    asm volatile("red.global.add.v2.f32 [%0+%3], {%1, %2};" ::"l"(base), "f"(__uint_as_float(a)),
                 "f"(__uint_as_float(b)), "n"(kOffBytes) : "memory");
}
template <int kOffBytes>
__device__ __forceinline__ void red_add_v4_at(float* base, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("red.global.add.v4.f32 [%0+%5], {%1, %2, %3, %4};" ::"l"(base), "f"(__uint_as_float(a)),
                 "f"(__uint_as_float(b)), "f"(__uint_as_float(c)), "f"(__uint_as_float(d)), "n"(kOffBytes)
                 : "memory");
}
// 16 consecutive queries of one head-dimension element into the interleaved
// accumulator ([groups of 4 queries][D][4]): g0 points at slot 0 of the group
// holding the first query, which sits in slot O.  Whole groups take one
// 16-byte reduction (a warp's 32 elements: 512 contiguous bytes), the partial
// groups at both ends 8- and 4-byte ones.
template <int D, int O>
__device__ __forceinline__ void red_add_run16(float* g0, const uint32_t (&v)[16]) {
    constexpr int kG = 16 * D;  // bytes between consecutive groups
    if constexpr (O == 0) {
        red_add_v4_at<0>(g0, v[0], v[1], v[2], v[3]);
        red_add_v4_at<kG>(g0, v[4], v[5], v[6], v[7]);
        red_add_v4_at<2 * kG>(g0, v[8], v[9], v[10], v[11]);
        red_add_v4_at<3 * kG>(g0, v[12], v[13], v[14], v[15]);
    } else if constexpr (O == 1) {
        red_add_f32_at<4>(g0, __uint_as_float(v[0]));
        red_add_v2_at<8>(g0, v[1], v[2]);
        red_add_v4_at<kG>(g0, v[3], v[4], v[5], v[6]);
        red_add_v4_at<2 * kG>(g0, v[7], v[8], v[9], v[10]);
        red_add_v4_at<3 * kG>(g0, v[11], v[12], v[13], v[14]);
        red_add_f32_at<4 * kG>(g0, __uint_as_float(v[15]));
    } else if constexpr (O == 2) {
        red_add_v2_at<8>(g0, v[0], v[1]);
        red_add_v4_at<kG>(g0, v[2], v[3], v[4], v[5]);
        red_add_v4_at<2 * kG>(g0, v[6], v[7], v[8], v[9]);
        red_add_v4_at<3 * kG>(g0, v[10], v[11], v[12], v[13]);
        red_add_v2_at<4 * kG>(g0, v[14], v[15]);
    } else {
        red_add_f32_at<12>(g0, __uint_as_float(v[0]));
        red_add_v4_at<kG>(g0, v[1], v[2], v[3], v[4]);
        red_add_v4_at<2 * kG>(g0, v[5], v[6], v[7], v[8]);
        red_add_v4_at<3 * kG>(g0, v[9], v[10], v[11], v[12]);
        red_add_v2_at<4 * kG>(g0, v[13], v[14]);
        red_add_f32_at<4 * kG + 8>(g0, __uint_as_float(v[15]));
    }
}

// Pairs (-LSE * log2(e), Delta = rowsum(dO * O)), head-major [Hq, pitch, 2]:
// rows < T from the forward, rows [T, T_cap) zero (they are only read for
// query columns that the backward masks).  The fp32 dQ accumulator ([Hq,
// pitch / 4, D, 4]: four consecutive queries interleaved per head-dimension
// element) is zeroed for the query groups that hold rows < T.
__global__ void attn_bwd_prep_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                                     const float* __restrict__ lse, const int32_t* __restrict__ total_tokens,
                                     int64_t T_cap, int64_t pitch, int Hq, int D, float2* __restrict__ lse_delta,
                                     float* __restrict__ dq_accum) {
    // one (token, head) row per group of D / 8 lanes, one 16-byte vector of O
    // and of dO per lane
    const int G = D >> 3;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t row = tid / G;
    const int part = (int)(tid - row * G);
    const int64_t T = min((int64_t)total_tokens[0], T_cap);
    const bool valid = row < T * Hq;
    float s = 0.f;
    if (valid) {
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(o + row * D) + part);
        const uint4 y = __ldg(reinterpret_cast<const uint4*>(dout + row * D) + part);
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s += __uint_as_float(xs[i] << 16) * __uint_as_float(ys[i] << 16);
            s += __uint_as_float(xs[i] & 0xffff0000u) * __uint_as_float(ys[i] & 0xffff0000u);
        }
    }
    // zero the accumulator: head h's groups [0, ceil(T / 4)) are 4 * D floats
    // each, contiguous; this thread's index covers two 16-byte vectors
    {
        const int64_t G4 = (T + 3) >> 2;
        const int64_t per_head = G4 * D / 2;  // vector pairs per head
        if (tid < per_head * Hq) {
            const int64_t h = tid / per_head;
            const int64_t k = tid - h * per_head;
            float4* acc = reinterpret_cast<float4*>(dq_accum + h * pitch * D) + 2 * k;
            acc[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    // reduce over the row's lanes (groups of G consecutive lanes, G a power of two)
    for (int off = G >> 1; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (part == 0 && row < T_cap * Hq) {
        const int64_t t = row / Hq;
        const int h = (int)(row - t * Hq);
        lse_delta[(int64_t)h * pitch + t] = valid ? make_float2(-lse[row] * kLog2e, s) : make_float2(0.f, 0.f);
    }
}

// dQ [T, Hq, D] = scale * accumulator [Hq, pitch / 4, D, 4], bf16, rows < T.
// A thread takes one group of four queries and eight head-dimension elements:
// 128 contiguous accumulator bytes in, four 16-byte bf16 rows out
__device__ __forceinline__ float comp4(const float4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}
__global__ void attn_dq_convert_kernel(const float* __restrict__ dq_accum, const int32_t* __restrict__ total_tokens,
                                       int64_t T_cap, int64_t pitch, int Hq, int D, float scale,
                                       __nv_bfloat16* __restrict__ dq) {
    const int d8 = D / 8;
    const int64_t T = min((int64_t)total_tokens[0], T_cap);
    const int64_t G4 = (T + 3) >> 2;
    const int64_t n = (int64_t)Hq * G4 * d8;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t hg = i / d8;  // (head, group), head-major
        const int c = (int)(i - hg * d8);
        const int64_t h = hg / G4;
        const int64_t g = hg - h * G4;
        const float4* src = reinterpret_cast<const float4*>(dq_accum + ((h * (pitch >> 2) + g) * D + 8 * c) * 4);
        float4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __ldg(src + k);
#pragma unroll
        for (int qi = 0; qi < 4; ++qi) {
            const int64_t t = 4 * g + qi;
            if (t >= T) break;
            uint4 w;
            w.x = pack_bf16x2(comp4(v[0], qi) * scale, comp4(v[1], qi) * scale);
            w.y = pack_bf16x2(comp4(v[2], qi) * scale, comp4(v[3], qi) * scale);
            w.z = pack_bf16x2(comp4(v[4], qi) * scale, comp4(v[5], qi) * scale);
            w.w = pack_bf16x2(comp4(v[6], qi) * scale, comp4(v[7], qi) * scale);
            *reinterpret_cast<uint4*>(dq + (t * Hq + h) * D + 8 * c) = w;
        }
    }
}

struct BwdParams {
    const KTile* ktiles;
    const int* counts;
    const int* kgroup_off;
    const int32_t* resp_off;
    const int32_t* resp_len;
    const int2* rblocks;
    int B;
    int Hq, Hkv, ratio;
    int64_t T_cap;
    const float2* lse_delta;  // [Hq, ld_pitch] (-LSE * log2(e), Delta)
    int64_t ld_pitch;
    float* dq_accum;   // [Hq, pitch / 4, D, 4] fp32: four consecutive queries per element
    int64_t acc_groups;  // pitch / 4: query groups per head
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    float scale;
    float scale_log2;
    int* status;
    int* sched;       // global unit counter (zeroed by the plan kernel)
    long long limit;
    int withhold;     // test option: the K/V load of unit 0 is skipped
};

template <int D>
struct BwdCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kTile = 128 * D * 2;
    // Q and dO are staged per 64-query half: a half-slot holds Q_h then dO_h,
    // each kChunks chunks of 64 rows x 64 columns (8 KB, 128-byte swizzle)
    static constexpr int kHalfChunk = 64 * 128;
    static constexpr int kHalf = 64 * D * 2;
    static constexpr int kStages = D == 128 ? 4 : 8;  // half-slots
    // dS of one half for the dQ GEMM: 128 key rows x 64 query columns, bf16,
    // 128-byte swizzle (one chunk)
    static constexpr int kDS = 128 * 128;
    // kfull, kempty, qfull[S], qempty[S], sfull[2], dpfull[2], pdsfull[2],
    // dqfull[2], dqfree[2], unit ring (4), mma drain
    static constexpr int kNumBars = 2 + 2 * kStages + 10 + 4 + 1;
    static constexpr int kDataBytes = 2 * kTile + kStages * 2 * kHalf + 2 * kDS;
    // per half-slot, beside Q and dO: the half's -LSE * log2(e) and Delta as
    // four 16-query chunks of 128 bytes (16 -LSE values, then 16 Delta
    // values), so that a softmax warp reads its chunk with 16-byte broadcast
    // loads, and the half's block descriptor {q0, nq, query head, diagonal}
    static constexpr int kLdStride = 512;
    static constexpr int kMetaBytes = 16;
    // data, LSE/Delta slots, descriptors, barriers, misc words; the dynamic
    // shared memory base is 1024-aligned (checked at run time)
    static constexpr int kSmemBytes = kDataBytes + kStages * (kLdStride + kMetaBytes) + kNumBars * 8 + 64;
    // TMEM: dV [0, D), dK [D, 2D); query half h: S^T [2D + 128h, +64) and
    // dP^T [2D + 128h + 64, +64).  The softmax writes P^T and dS^T (bf16 pairs)
    // back over the S^T columns it read; dQ^T of the half (fp32, lanes = head
    // dimension) goes into the dP^T columns once the softmax has read them.
    static constexpr uint32_t kColV = 0, kColK = D;
    __host__ __device__ static constexpr uint32_t col_s(int h) { return 2 * D + 128 * h; }
    __host__ __device__ static constexpr uint32_t col_p(int h) { return 2 * D + 128 * h + 64; }
};
static_assert(BwdCfg<128>::kSmemBytes <= 232448, "shared memory of the D = 128 backward");
static_assert(BwdCfg<64>::kSmemBytes <= 232448, "shared memory of the D = 64 backward");

struct QBlock {
    int q0, nq;
    bool diag;
};

// idx-th query block that sees key tile t (see the file comment for the order):
// the prompt's own blocks from the diagonal on, then (prompt key tiles) every
// response block of the group from the plan's list.
__device__ __forceinline__ QBlock qblock_of(const KTile& t, const BwdParams& p, int idx, int rb_base) {
    QBlock qb;
    if (t.kind == 0) {
        const int plen = t.pk1 - t.pk0;
        const int jt = (t.k0 - t.pk0) >> 7;
        const int npt = cdiv128(plen);
        if (idx < npt - jt) {
            const int i = jt + idx;
            qb.q0 = t.pk0 + 128 * i;
            qb.nq = min(128, plen - 128 * i);
            qb.diag = (i == jt);
            return qb;
        }
        const int2 e = p.rblocks[rb_base + idx - (npt - jt)];
        qb.q0 = e.x;
        qb.nq = e.y;
        qb.diag = false;
        return qb;
    }
    const int roff = p.resp_off[t.b], rlen = p.resp_len[t.b];
    const int jt = (t.k0 - roff) >> 7;
    const int i = jt + idx;
    qb.q0 = roff + 128 * i;
    qb.nq = min(128, rlen - 128 * i);
    qb.diag = (i == jt);
    return qb;
}


// producer warp, MMA-issuer warp, then 4 softmax warpgroups (warps 2-17; a
// warpgroup's four warps still cover the four TMEM lane quarters, warp & 3)
constexpr int kBwdThreads = 576;

// Each 128-query block is processed as two 64-query halves A and B with their
// own TMEM columns, so that one half's softmax overlaps the other half's GEMMs.
// MMA order per block `it` (waits in brackets):
//   S^T_A | [dQ^T_A(it-1) read out] dP^T_A | [softmax B(it-1)] dQ^T, dV, dK of B(it-1)
//   | S^T_B | [dQ^T_B(it-1) read out] dP^T_B | [softmax A(it)] dQ^T, dV, dK of A(it)
// The softmax warps run: softmax A(it) | read out dQ^T_B(it-1) | softmax B(it)
// | read out dQ^T_A(it).  The four warpgroups take 16 query columns of a half
// each (warpgroup g: columns [16 g, +16)); a warpgroup writes P^T and dS^T
// (bf16 pairs, 8 columns each) over the 16 S^T columns it read, which are the
// A operands of K step g of dV += P^T dO and dK += dS^T Q.  dS also goes to
// shared memory as the B operand of dQ^T = K^T dS^T.  MMAs of one thread
// complete in order, so S^T of the next block may overwrite columns that the
// accumulations of the previous one read.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const BwdParams p) {
    using C = BwdCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t s0 = smem_u32(smem);
    if (s0 & 1023) {  // the 128-byte swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) atomicCAS(p.status, 0, 1099);
        return;
    }
    const uint32_t sK = s0, sV = s0 + C::kTile;
    const uint32_t sQD = s0 + 2 * C::kTile;  // half-slot s: Q_h at sQD + s*2*kHalf, dO_h at + kHalf
    const uint32_t sDS = sQD + C::kStages * 2 * C::kHalf;  // half h at sDS + h*kDS
    const uint32_t sLD = s0 + C::kDataBytes;                   // slot s: chunks at sLD + s*kLdStride
    const uint32_t sMeta = sLD + C::kStages * C::kLdStride;    // slot s: int4 at sMeta + 16 s
    const uint32_t bar0 = sMeta + C::kStages * C::kMetaBytes;
    const uint32_t b_kfull = bar0, b_kempty = bar0 + 8;
    auto b_qfull = [&](int s) { return bar0 + 16 + 8 * s; };
    auto b_qempty = [&](int s) { return bar0 + 16 + 8 * (C::kStages + s); };
    const uint32_t b_rest = bar0 + 16 + 16 * C::kStages;
    auto b_sfull = [&](int h) { return b_rest + 8 * h; };
    auto b_dpfull = [&](int h) { return b_rest + 16 + 8 * h; };
    auto b_pdsfull = [&](int h) { return b_rest + 32 + 8 * h; };
    auto b_dqfull = [&](int h) { return b_rest + 48 + 8 * h; };
    auto b_dqfree = [&](int h) { return b_rest + 64 + 8 * h; };
    uint8_t* misc = smem + (bar0 - s0) + C::kNumBars * 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 8);
    const UnitRing ring{b_rest + 80, b_rest + 96, reinterpret_cast<volatile int*>(misc + 16)};
    const uint32_t b_drain = b_rest + 112;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(b_drain, 1);
        mbar_init(b_kfull, 1);
        mbar_init(b_kempty, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(b_qfull(s), 1);
            mbar_init(b_qempty(s), 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(b_sfull(h), 1);
            mbar_init(b_dpfull(h), 1);
            mbar_init(b_pdsfull(h), 16);  // one arrival per softmax warp
            mbar_init(b_dqfull(h), 1);
            mbar_init(b_dqfree(h), 16);
        }
        ring_init(ring, 17);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const AbortState ab{abort_flag, p.status, p.limit};
    const int n_units = p.counts[1] * p.Hkv;

    if (warp == 0) {
        // producer: the whole warp runs the loop (warp-uniform control); lane 0
        // takes the units and issues the copies, and every lane stages two
        // query columns of a half's -LSE/Delta chunks (lane l: chunk l / 8,
        // columns 2 (l % 8) and 2 (l % 8) + 1)
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_do);
        }
        const int lcol = 16 * (lane >> 3) + 2 * (lane & 7);
        const uint32_t lofs = 128 * (lane >> 3) + 8 * (lane & 7);
        int qstage = 0, k = 0, last_k = -1;
        bool ok = true;
        for (; ok; ++k) {
            int u = 0;
            if (lane == 0) u = ring_publish(ring, k, p.sched, n_units, ab);
            u = __shfl_sync(0xffffffffu, u, 0);
            if (u < 0) { ok = (u == -1); break; }
            int ti, hk;
            decode_unit(u, p.kgroup_off, p.B, p.Hkv, ti, hk);
            const KTile t = p.ktiles[ti];
            if (k > 0 && !__all_sync(0xffffffffu, mbar_wait(b_kempty, (k - 1) & 1, ab, 31))) { ok = false; break; }
            // test option: the CTA that takes unit 0 withholds its K/V load, so
            // that a bounded wait runs out and the abort path runs
            if (!(p.withhold && u == 0)) {
                if (lane == 0) {
                    mbar_expect_tx(b_kfull, 2 * C::kTile);
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c) {
                        tma_load_2d(sK + c * kChunkBytes, &tm_k, hk * D + 64 * c, t.k0, b_kfull);
                        tma_load_2d(sV + c * kChunkBytes, &tm_v, hk * D + 64 * c, t.k0, b_kfull);
                    }
                }
                last_k = k;
            }
            const int rb_base = t.kind == 0 ? p.kgroup_off[t.g] : 0;
            for (int hh = 0; hh < p.ratio && ok; ++hh) {
                const int h = hk * p.ratio + hh;
                const float2* ld_h = p.lse_delta + (int64_t)h * p.ld_pitch;
                for (int qi = 0; qi < t.nqblk && ok; ++qi) {
                    const QBlock qb = qblock_of(t, p, qi, rb_base);
                    for (int half = 0; half < 2; ++half) {
                        const int slot = qstage % C::kStages, r = qstage / C::kStages;
                        if (r > 0 && !__all_sync(0xffffffffu, mbar_wait(b_qempty(slot), (r - 1) & 1, ab, 32))) {
                            ok = false;
                            break;
                        }
                        const int row = qb.q0 + 64 * half;
                        // this lane's two columns (rows past T_cap: zero; the softmax
                        // masks every column past the block's queries)
                        const int c0 = row + lcol;
                        const float2 va = c0 < p.T_cap ? ld_h[c0] : make_float2(0.f, 0.f);
                        const float2 vb = c0 + 1 < p.T_cap ? ld_h[c0 + 1] : make_float2(0.f, 0.f);
                        const uint32_t dst = sLD + slot * C::kLdStride + lofs;
                        st_shared_v2(dst, va.x, vb.x);
                        st_shared_v2(dst + 64, va.y, vb.y);
                        // the lanes' stores, then lane 0's descriptor, precede its
                        // arrival (release) that the consumers acquire
                        __syncwarp();
                        if (lane == 0) {
                            st_shared_v4_nc(sMeta + slot * C::kMetaBytes, (uint32_t)qb.q0, (uint32_t)qb.nq,
                                            (uint32_t)h, qb.diag ? 1u : 0u);
                            mbar_expect_tx(b_qfull(slot), 2 * C::kHalf);
                            const uint32_t qb_s = sQD + slot * 2 * C::kHalf;
                            // one box per tensor: 64 rows x the head's kChunks column chunks
                            tma_load_3d(qb_s, &tm_q, 0, row, h * C::kChunks, b_qfull(slot));
                            tma_load_3d(qb_s + C::kHalf, &tm_do, 0, row, h * C::kChunks, b_qfull(slot));
                        }
                        ++qstage;
                    }
                }
            }
        }
        if (lane == 0) {
            const long long lim = p.limit;
            if (ok) {
                // every load consumed and every release committed before exit
                for (int s = qstage - C::kStages; s < qstage; ++s)
                    if (s >= 0) mbar_wait_drain(b_qempty(s % C::kStages), (s / C::kStages) & 1, lim);
                if (k > 0) mbar_wait_drain(b_kempty, (k - 1) & 1, lim);
            } else {
                // abort: the consumers have left; wait until the copies in flight landed
                for (int s = qstage - C::kStages; s < qstage; ++s)
                    if (s >= 0) mbar_wait_drain(b_qfull(s % C::kStages), (s / C::kStages) & 1, lim);
                if (last_k >= 0) mbar_wait_drain(b_kfull, last_k & 1, lim);
            }
        }
    } else if (warp == 1) {
        // the whole warp runs the issue loop (warp-uniform state); the elected
        // lane executes the tcgen05 instructions
        const bool leader = elect_one_sync();
        auto wait = [&](uint32_t bar, uint32_t parity, int where) {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, ab, where));
        };
        constexpr uint32_t idesc_s = idesc_bf16_f32(128, 64, false, false);
        constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, false, true);
        constexpr uint32_t idesc_dq = idesc_bf16_f32(128, 64, true, true);
        int qstage = 0, k = 0, pds_cnt[2] = {0, 0}, dq_cnt[2] = {0, 0};
        bool ok = true;
        // base descriptors; a K step adds a compile-time offset (in 16-byte
        // units) to the start-address field, which never carries out of it
        const uint64_t dK0 = smem_desc(sK, 16, 1024), dV0 = smem_desc(sV, 16, 1024);
        // K^T as the A operand of dQ^T (M = head dimension, MN-major; for D = 64
        // rows 64-127 read the V tile and land in TMEM lanes nobody reads)
        const uint64_t dKt0 = smem_desc(sK, kChunkBytes, 1024);
        // S^T_h = K Q_h^T for query half h (half-slot `slot`)
        auto issue_s = [&](int slot, int h) {
            const uint64_t dq0 = smem_desc(sQD + slot * 2 * C::kHalf, 16, 1024);
#pragma unroll
            for (int s = 0; s < D / 16; ++s) {
                const uint32_t ka = ((s >> 2) * kChunkBytes + (s & 3) * 32) >> 4;
                const uint32_t qa = ((s >> 2) * C::kHalfChunk + (s & 3) * 32) >> 4;
                if (leader) mma_bf16_ss(tmem + C::col_s(h), dK0 + ka, dq0 + qa, idesc_s, s > 0 ? 1u : 0u);
            }
            if (leader) mma_commit(b_sfull(h));
        };
        // dP^T_h = V dO_h^T, once the previous dQ^T_h (same columns) was read out
        auto issue_dp = [&](int slot, int h) -> bool {
            if (dq_cnt[h] > 0 && !wait(b_dqfree(h), (dq_cnt[h] - 1) & 1, 37)) return false;
            tc_fence_after();
            const uint64_t ddo0 = smem_desc(sQD + slot * 2 * C::kHalf + C::kHalf, 16, 1024);
#pragma unroll
            for (int s = 0; s < D / 16; ++s) {
                const uint32_t ka = ((s >> 2) * kChunkBytes + (s & 3) * 32) >> 4;
                const uint32_t qa = ((s >> 2) * C::kHalfChunk + (s & 3) * 32) >> 4;
                if (leader) mma_bf16_ss(tmem + C::col_p(h), dV0 + ka, ddo0 + qa, idesc_s, s > 0 ? 1u : 0u);
            }
            if (leader) mma_commit(b_dpfull(h));
            return true;
        };
        // once the softmax wrote half h: dQ^T_h = K^T dS^T_h (B from shared
        // memory) into the dP^T columns, then dV += P^T_h dO_h and dK += dS^T_h
        // Q_h (A operands from TMEM; first = overwrite)
        auto issue_acc = [&](int slot, int h, bool first) -> bool {
            if (!wait(b_pdsfull(h), pds_cnt[h] & 1, 35)) return false;
            ++pds_cnt[h];
            tc_fence_after();
            // dQ^T first, so that its read-out (which frees the dP^T columns for
            // the next block) overlaps the dV and dK GEMMs
            const uint64_t dds0 = smem_desc(sDS + h * C::kDS, C::kDS, 1024);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                if (leader) mma_bf16_ss(tmem + C::col_p(h), dKt0 + s * 128, dds0 + s * 128, idesc_dq, s > 0 ? 1u : 0u);
            if (leader) mma_commit(b_dqfull(h));
            ++dq_cnt[h];
            const uint32_t qh = sQD + slot * 2 * C::kHalf, dh = qh + C::kHalf;
            const uint64_t bq0 = smem_desc(qh, C::kHalfChunk, 1024), bdo0 = smem_desc(dh, C::kHalfChunk, 1024);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                if (leader) mma_bf16_ts(tmem + C::kColV, tmem + C::col_s(h) + 16 * s, bdo0 + s * 128, idesc_acc,
                                        (!first || s > 0) ? 1u : 0u);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                if (leader) mma_bf16_ts(tmem + C::kColK, tmem + C::col_s(h) + 16 * s + 8, bq0 + s * 128, idesc_acc,
                                        (!first || s > 0) ? 1u : 0u);
            return true;
        };
        for (; ok; ++k) {
            const int u = ring_take_warp(ring, k, ab);
            if (u < 0) { ok = (u == -1); break; }
            int ti, hk;
            decode_unit(u, p.kgroup_off, p.B, p.Hkv, ti, hk);
            const int iters = p.ktiles[ti].nqblk * p.ratio;
            if (!wait(b_kfull, k & 1, 33)) { ok = false; break; }
            tc_fence_after();
            int prev_b = -1;  // half-slot of the previous block's half B
            for (int it = 0; it < iters && ok; ++it) {
                const int slot_a = qstage % C::kStages;
                if (!wait(b_qfull(slot_a), (qstage / C::kStages) & 1, 34)) { ok = false; break; }
                ++qstage;
                tc_fence_after();
                issue_s(slot_a, 0);
                if (!issue_dp(slot_a, 0)) { ok = false; break; }
                if (it > 0) {
                    if (!issue_acc(prev_b, 1, false)) { ok = false; break; }
                    if (leader) mma_commit(b_qempty(prev_b));
                }
                const int slot_b = qstage % C::kStages;
                if (!wait(b_qfull(slot_b), (qstage / C::kStages) & 1, 34)) { ok = false; break; }
                ++qstage;
                tc_fence_after();
                issue_s(slot_b, 1);
                if (!issue_dp(slot_b, 1)) { ok = false; break; }
                if (!issue_acc(slot_a, 0, it == 0)) { ok = false; break; }
                if (leader) mma_commit(b_qempty(slot_a));
                prev_b = slot_b;
            }
            if (!ok) break;
            if (!issue_acc(prev_b, 1, false)) { ok = false; break; }
            if (leader) mma_commit(b_qempty(prev_b));
            if (leader) mma_commit(b_kempty);  // every MMA of the unit done: K/V reusable, dV/dK final
        }
        drain_mmas(leader, b_drain, p.limit);
    } else {
        // softmax warps: warpgroup wg owns query columns [16 wg, +16) of each
        // 64-query half; all four warpgroups take half A, then half B.  TMEM
        // lane r is key row r of S^T / dP^T and head-dimension row r of dQ^T.
        // The query block, its head and its LSE/Delta come from the half-slot
        // (written by the producer), so the loop reads no global memory.
        const int wg = (warp - 2) >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
        const float sl2 = p.scale_log2;
        int s_cnt[2] = {0, 0}, dp_cnt[2] = {0, 0}, rd_cnt[2] = {0, 0};
        int qstage = 0;  // half-slot sequence, as the producer and the MMA warp run it
        bool ok = true;
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        // dQ^T of half hf of block qb (query head h): this warpgroup's 16 query
        // columns, added into the fp32 accumulator; lanes are head-dim rows, so
        // a warp's adds for one query cover 32 consecutive floats
        auto readout = [&](int hf, const QBlock& qb, int h) -> bool {
            if (!__all_sync(0xffffffffu, mbar_wait(b_dqfull(hf), rd_cnt[hf] & 1, ab, 39))) return false;
            ++rd_cnt[hf];
            tc_fence_after();
            uint32_t v[16];
            tmem_ld16(trow + C::col_p(hf) + 16 * wg, v);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(b_dqfree(hf));
            const int qlo = 64 * hf + 16 * wg;
            const int nv = qb.nq - qlo;
            if (r < D && qlo < qb.nq &&
                ZR_BOUNDS(qb.q0 + qlo + min(nv, 16) <= p.T_cap, p.status - kStatusTimeout, 20)) {
                // element (query q, row r) of head h sits at group q / 4, slot q % 4
                const int q = qb.q0 + qlo;  // first of the 16 query columns
                float* head = p.dq_accum + ((int64_t)h * p.acc_groups * D + r) * 4;
                if (nv >= 16) {
                    float* g0 = head + (int64_t)(q >> 2) * D * 4;
                    switch (q & 3) {  // warp-uniform
                        case 0: red_add_run16<D, 0>(g0, v); break;
                        case 1: red_add_run16<D, 1>(g0, v); break;
                        case 2: red_add_run16<D, 2>(g0, v); break;
                        default: red_add_run16<D, 3>(g0, v); break;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (j < nv) red_add_f32(head + (int64_t)((q + j) >> 2) * D * 4 + ((q + j) & 3),
                                                __uint_as_float(v[j]));
                }
            }
            return true;
        };
        for (int k = 0; ok; ++k) {
            const int u = ring_take_warp(ring, k, ab);
            if (u < 0) { ok = (u == -1); break; }
            int ti, hk;
            decode_unit(u, p.kgroup_off, p.B, p.Hkv, ti, hk);
            const KTile t = p.ktiles[ti];
            const int key_pos = t.k0 + r;
            const bool key_ok = r < t.nk;  // rows past the tile's keys give no dS (they feed dQ)
            const int iters = t.nqblk * p.ratio;
            QBlock qb_prev{0, 0, false};
            int h_prev = 0;
            for (int it = 0; it < iters && ok; ++it) {
                QBlock qb{0, 0, false};
                int h_cur = 0;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int slot = qstage % C::kStages;
                    const uint32_t qph = (uint32_t)(qstage / C::kStages) & 1u;
                    ++qstage;
                    if (!__all_sync(0xffffffffu, mbar_wait(b_sfull(hf), s_cnt[hf] & 1, ab, 36))) {
                        ok = false;
                        break;
                    }
                    ++s_cnt[hf];
                    tc_fence_after();
                    uint32_t sr[16];
                    tmem_ld16(trow + C::col_s(hf) + 16 * wg, sr);
                    // the slot was filled before S^T was issued; this wait completes
                    // at once and makes the producer's descriptor and pairs visible
                    if (!__all_sync(0xffffffffu, mbar_wait(b_qfull(slot), qph, ab, 41))) {
                        ok = false;
                        break;
                    }
                    if (hf == 0) {
                        const int4 m = *reinterpret_cast<const int4*>(smem + (sMeta - s0) + slot * C::kMetaBytes);
                        qb.q0 = m.x;
                        qb.nq = m.y;
                        h_cur = m.z;
                        qb.diag = m.w != 0;
                    }
                    const int row0 = qb.q0 + 64 * hf;
                    // -LSE * log2(e) (16 floats), then Delta (16 floats), of this
                    // warpgroup's 16 query columns
                    const float4* ldc =
                        reinterpret_cast<const float4*>(smem + (sLD - s0) + slot * C::kLdStride + 128 * wg);
                    const int nv = qb.nq - 64 * hf - 16 * wg;  // valid query columns of this warpgroup
                    tmem_wait_ld();
                    // P^T from S^T and the staged LSE
                    const int qlo = key_ok ? key_pos - row0 - 16 * wg : (1 << 30);  // causal: query >= key
                    float pv[16];
                    auto probs = [&](auto masked) {
                        constexpr bool kMasked = decltype(masked)::value;
#pragma unroll
                        for (int pc = 0; pc < 8; ++pc) {
                            // S * scale * log2(e) - LSE * log2(e), two columns per instruction
                            const float4 l4 = ldc[pc >> 1];
                            float x[2];
                            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * pc]), __uint_as_float(sr[2 * pc + 1])),
                                             sl2x2, (pc & 1) ? f2_pack(l4.z, l4.w) : f2_pack(l4.x, l4.y)),
                                      x[0], x[1]);
#pragma unroll
                            for (int i = 0; i < 2; ++i) {
                                const int col = 2 * pc + i;
                                float pr = ex2(x[i]);
                                if (kMasked) pr = (col >= qlo && col < nv) ? pr : 0.f;
                                pv[col] = pr;
                            }
                        }
                    };
                    if (qb.diag || !key_ok || nv < 16) probs(std::integral_constant<bool, true>());
                    else probs(std::integral_constant<bool, false>());
                    // dS^T from dP^T and the staged Delta
                    if (!__all_sync(0xffffffffu, mbar_wait(b_dpfull(hf), dp_cnt[hf] & 1, ab, 38))) {
                        ok = false;
                        break;
                    }
                    ++dp_cnt[hf];
                    tc_fence_after();
                    uint32_t dr[16];
                    tmem_ld16(trow + C::col_p(hf) + 16 * wg, dr);
                    tmem_wait_ld();
                    uint32_t pd[16];  // P^T (8 bf16 pairs), then dS^T (8 pairs)
#pragma unroll
                    for (int pc = 0; pc < 8; ++pc) {
                        // dS = P * (dP - Delta), two columns per instruction (the
                        // staged Delta of a masked column is finite, so its dS is 0)
                        const float4 d4 = ldc[4 + (pc >> 1)];
                        float ds[2];
                        f2_unpack(f2_mul(f2_pack(pv[2 * pc], pv[2 * pc + 1]),
                                         f2_sub(f2_pack(__uint_as_float(dr[2 * pc]), __uint_as_float(dr[2 * pc + 1])),
                                                (pc & 1) ? f2_pack(d4.z, d4.w) : f2_pack(d4.x, d4.y))),
                                  ds[0], ds[1]);
                        pd[pc] = pack_bf16x2(pv[2 * pc], pv[2 * pc + 1]);
                        pd[8 + pc] = pack_bf16x2(ds[0], ds[1]);
                    }
                    // P^T and dS^T (bf16 pairs) over the 16 S^T columns read, one store
                    tmem_st16(trow + C::col_s(hf) + 16 * wg, pd);
                    // dS into shared memory, key row r, query columns [16 wg, +16):
                    // 16-byte pieces 2 wg and 2 wg + 1 of the row, 128-byte swizzle.
                    // The previous dQ^T of this half, which read the buffer, has
                    // completed: its result was read out before this half began.
                    {
                        const uint32_t row = sDS + hf * C::kDS + (r >> 3) * 1024 + (r & 7) * 128;
                        st_shared_v4_nc(row + (((2 * wg) ^ (r & 7)) << 4), pd[8], pd[9], pd[10], pd[11]);
                        st_shared_v4_nc(row + (((2 * wg + 1) ^ (r & 7)) << 4), pd[12], pd[13], pd[14], pd[15]);
                    }
                    fence_async_smem();
                    tmem_wait_st();
                    tc_fence_before();
                    // every lane's TMEM and shared-memory writes (and its reads of
                    // the slot) precede the warp's one arrival
                    __syncwarp();
                    if (lane == 0) mbar_arrive(b_pdsfull(hf));
                    // the other half's dQ^T, issued after this half's GEMMs began
                    if (hf == 0 && it > 0) {
                        if (!readout(1, qb_prev, h_prev)) { ok = false; break; }
                    } else if (hf == 1) {
                        if (!readout(0, qb, h_cur)) { ok = false; break; }
                    }
                }
                qb_prev = qb;
                h_prev = h_cur;
            }
            if (!ok) break;
            if (!readout(1, qb_prev, h_prev)) { ok = false; break; }
            // epilogue: every MMA of unit k is done once its kempty phase completed (the
            // MMA thread commits it after the unit's last accumulation; the next unit
            // cannot finish before this epilogue, so the phase parity is unambiguous).
            // Warpgroups 0-1 write dV columns [64 wg, +64), 2-3 write scale * dK.
            if (!__all_sync(0xffffffffu, mbar_wait(b_kempty, k & 1, ab, 40))) { ok = false; break; }
            tc_fence_after();
            const bool store = r < t.nk && ZR_BOUNDS(key_pos < p.T_cap, p.status - kStatusTimeout, 21);
            const bool is_k = wg >= 2;
            const int c0 = 64 * (wg & 1);
            const uint32_t col = (is_k ? C::kColK : C::kColV) + c0;
            const float mul = is_k ? p.scale : 1.0f;
            __nv_bfloat16* out = (is_k ? p.dk : p.dv) + ((int64_t)key_pos * p.Hkv + hk) * D + c0;
            if (c0 < D) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t o[32];
                    tmem_ld32(trow + col + 32 * c, o);
                    tmem_wait_ld();
                    if (store) {
#pragma unroll
                        for (int i = 0; i < 32; i += 8) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(o[i + 0]) * mul, __uint_as_float(o[i + 1]) * mul);
                            w.y = pack_bf16x2(__uint_as_float(o[i + 2]) * mul, __uint_as_float(o[i + 3]) * mul);
                            w.z = pack_bf16x2(__uint_as_float(o[i + 4]) * mul, __uint_as_float(o[i + 5]) * mul);
                            w.w = pack_bf16x2(__uint_as_float(o[i + 6]) * mul, __uint_as_float(o[i + 7]) * mul);
                            *reinterpret_cast<uint4*>(out + 32 * c + i) = w;
                        }
                    }
                }
            }
            tc_fence_before();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D>
zr_status launch_bwd(const zr_recon_info& info, const AttnWorkspace& ws, const AttnArgs& a, cudaStream_t s) {
    using C = BwdCfg<D>;
    CUtensorMap tq, tk, tv, tdo;
    zr_status st;
    // Q and dO: [64-column chunk, row, chunk index] views, boxes of 64 rows x
    // the kChunks chunks of one head (the kernel stages them per 64-query
    // half, chunk-major, 128-byte swizzle)
    for (int w = 0; w < 2; ++w) {
        EncodeTiledFn fn = encode_fn();
        if (!fn) return set_error(ZR_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
        const void* base = w == 0 ? a.q : a.dout;
        const int64_t row_bytes = (int64_t)a.Hq * D * 2;
        if (((uintptr_t)base & 15) || (row_bytes & 15))
            return set_error(ZR_ERR_INVALID_ARG, "q/k/v must be 16-byte aligned with 16-byte row strides");
        cuuint64_t dims[3] = {64, (cuuint64_t)a.T_cap, (cuuint64_t)(a.Hq * D / 64)};
        cuuint64_t strides[2] = {(cuuint64_t)row_bytes, 128};
        cuuint32_t box[3] = {64, 64, (cuuint32_t)C::kChunks};
        cuuint32_t estr[3] = {1, 1, 1};
        const CUresult r = fn(w == 0 ? &tq : &tdo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return set_error(ZR_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    }
    if ((st = make_map(&tk, a.k, (int64_t)a.Hkv * D, a.T_cap, (int64_t)a.Hkv * D * 2)) != ZR_OK) return st;
    if ((st = make_map(&tv, a.v, (int64_t)a.Hkv * D, a.T_cap, (int64_t)a.Hkv * D * 2)) != ZR_OK) return st;
    if (((uintptr_t)a.dq & 15) || ((uintptr_t)ws.dq_accum & 15))
        return set_error(ZR_ERR_INVALID_ARG, "dq must be 16-byte aligned");
    {
        const int64_t threads = lse_delta_pitch(a.T_cap) * a.Hq * (D / 8);
        const int64_t blocks = (threads + 255) / 256;
        KernelTimer timer("attn_bwd_prep", s);
        attn_bwd_prep_kernel<<<(unsigned)blocks, 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(a.o_in), static_cast<const __nv_bfloat16*>(a.dout), a.lse_in,
            info.total_tokens, a.T_cap, lse_delta_pitch(a.T_cap), a.Hq, D, ws.lse_delta, ws.dq_accum);
        ZR_LAUNCH_CHECK("attn_bwd_prep_kernel");
    }
    BwdParams p;
    p.ktiles = ws.plan.ktiles;
    p.counts = ws.plan.counts;
    p.kgroup_off = ws.plan.group_ktile_off;
    p.resp_off = info.resp_off;
    p.resp_len = info.resp_len;
    p.rblocks = ws.plan.rblocks;
    p.B = info.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.ratio = a.Hq / a.Hkv;
    p.T_cap = a.T_cap;
    p.lse_delta = ws.lse_delta;
    p.ld_pitch = lse_delta_pitch(a.T_cap);
    p.dq_accum = ws.dq_accum;
    p.acc_groups = lse_delta_pitch(a.T_cap) / 4;
    p.dk = static_cast<__nv_bfloat16*>(a.dk);
    p.dv = static_cast<__nv_bfloat16*>(a.dv);
    p.scale = a.scale;
    p.scale_log2 = a.scale * kLog2e;
    p.status = info.status + kStatusTimeout;  // read by zr_check_status(info)
    p.sched = ws.plan.counts + 3;
    p.limit = wait_limit_cycles();
    p.withhold = (options().test_withhold & 2) != 0;
    ZR_CUDA_TRY(cudaFuncSetAttribute(attn_bwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::kSmemBytes));
    {
        KernelTimer timer("attn_bwd", s);
        attn_bwd_tc_kernel<D><<<num_sms(), kBwdThreads, C::kSmemBytes, s>>>(tq, tk, tv, tdo, p);
        ZR_LAUNCH_CHECK("attn_bwd_tc_kernel");
    }
    {
        KernelTimer timer("attn_dq_convert", s);
        attn_dq_convert_kernel<<<num_sms() * 8, 256, 0, s>>>(ws.dq_accum, info.total_tokens, a.T_cap,
                                                             lse_delta_pitch(a.T_cap), a.Hq, D,
                                                             a.scale, static_cast<__nv_bfloat16*>(a.dq));
        ZR_LAUNCH_CHECK("attn_dq_convert_kernel");
    }
    return ZR_OK;
}

}  // namespace

bool tc_bwd_supported(const AttnArgs& a) {
    return a.dtype == ZR_BF16 && (a.D == 64 || a.D == 128) && a.Hkv > 0 && a.Hq % a.Hkv == 0;
}

zr_status launch_attn_bwd_tc(const zr_recon_info& info, const AttnWorkspace& ws, const AttnArgs& a,
                             cudaStream_t s) {
    if (a.D == 128) return launch_bwd<128>(info, ws, a, s);
    return launch_bwd<64>(info, ws, a, s);
}

}  // namespace zr
