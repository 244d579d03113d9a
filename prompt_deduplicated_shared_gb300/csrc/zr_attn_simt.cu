// Split attention on CUDA cores (SIMT), forward and backward.
//
// This is the float32 path (float32 inputs and outputs, e.g. the 2-head,
// head_dim 64 parity configuration); bf16 attention runs only on the
// tensor-core kernels.  It computes the same split attention as those kernels
// ("How Prompt Deduplication Works", "Split Attention Optimization") from the
// same tile lists: a query tile of 128 rows attends the group's valid prompt
// [pk0, pk1) and the causal range [ck0, row].
//
// Layout: one warp owns a query (or key) row, its 32 lanes split the head
// dimension (DPL = D/32 values per lane); a block of 16 warps owns a 128-row
// tile and stages 32 keys (or queries) at a time in shared memory as fp32.
// Softmax runs in base 2 with the scale folded into log2(e).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "zr_internal.h"

namespace zr {
namespace {

constexpr int kWarps = 16;
constexpr int kRowsPerWarp = kTileM / kWarps;  // 8
constexpr int kChunk = 32;                      // keys / queries staged per step
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Key position kp of the virtual key index j of tile t: first the prefix
// [pk0, pk1), then the causal range from ck0.
__device__ __forceinline__ int key_pos(const QTile& t, int j) {
    const int np = t.pk1 - t.pk0;
    return j < np ? t.pk0 + j : t.ck0 + (j - np);
}

template <typename T, int DPL>
__global__ void __launch_bounds__(kWarps * 32)
attn_fwd_simt_kernel(const QTile* __restrict__ tiles, const int* __restrict__ counts,
                     const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     T* __restrict__ o, float* __restrict__ lse, int Hq, int Hkv,
                     float scale_log2) {
    constexpr int D = DPL * 32;
    __shared__ float sk[kChunk][D + 1];
    __shared__ float sv[kChunk][D];
    if ((int)blockIdx.x >= counts[0]) return;
    const QTile t = tiles[blockIdx.x];
    const int h = blockIdx.y;
    const int hk = h / (Hq / Hkv);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    float qr[kRowsPerWarp][DPL], acc[kRowsPerWarp][DPL], m[kRowsPerWarp], l[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int row = warp * kRowsPerWarp + r;
        const int64_t rp = t.q0 + min(row, t.nq - 1);
#pragma unroll
        for (int d = 0; d < DPL; ++d) {
            qr[r][d] = to_f(q[(rp * Hq + h) * D + lane + 32 * d]);
            acc[r][d] = 0.f;
        }
        m[r] = -INFINITY;
        l[r] = 0.f;
    }
    const int nkeys = (t.pk1 - t.pk0) + (t.q0 + t.nq - t.ck0);
    for (int j0 = 0; j0 < nkeys; j0 += kChunk) {
        __syncthreads();
        for (int i = threadIdx.x; i < kChunk * D; i += blockDim.x) {
            const int jj = i / D, d = i % D;
            const int j = j0 + jj;
            float kv = 0.f, vv = 0.f;
            if (j < nkeys) {
                const int64_t kp = key_pos(t, j);
                kv = to_f(k[(kp * Hkv + hk) * D + d]);
                vv = to_f(v[(kp * Hkv + hk) * D + d]);
            }
            sk[jj][d] = kv;
            sv[jj][d] = vv;
        }
        __syncthreads();
        const int jn = min(kChunk, nkeys - j0);
        for (int jj = 0; jj < jn; ++jj) {
            const int j = j0 + jj;
            const int kp = key_pos(t, j);
            const bool prefix = j < (t.pk1 - t.pk0);
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                const int row = warp * kRowsPerWarp + r;
                const int rp = t.q0 + row;
                if (!(prefix || kp <= rp)) continue;  // causal mask (warp-uniform)
                float s = 0.f;
#pragma unroll
                for (int d = 0; d < DPL; ++d) s += qr[r][d] * sk[jj][lane + 32 * d];
                s = warp_sum(s) * scale_log2;
                const float mn = fmaxf(m[r], s);
                const float alpha = exp2f(m[r] - mn);
                const float p = exp2f(s - mn);
                l[r] = l[r] * alpha + p;
#pragma unroll
                for (int d = 0; d < DPL; ++d) acc[r][d] = acc[r][d] * alpha + p * sv[jj][lane + 32 * d];
                m[r] = mn;
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int row = warp * kRowsPerWarp + r;
        if (row >= t.nq) continue;
        const int64_t rp = t.q0 + row;
        const float inv = 1.f / l[r];
#pragma unroll
        for (int d = 0; d < DPL; ++d) o[(rp * Hq + h) * D + lane + 32 * d] = from_f<T>(acc[r][d] * inv);
        if (lane == 0) lse[rp * Hq + h] = (m[r] + log2f(l[r])) * kLn2;
    }
}

// delta[row, h] = sum_d dO * O  (rows < T)
template <typename T>
__global__ void attn_delta_kernel(const T* __restrict__ o, const T* __restrict__ dout,
                                  const int32_t* __restrict__ total_tokens, int64_t T_cap, int Hq,
                                  int D, float* __restrict__ delta) {
    const int lane = threadIdx.x & 31;
    const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t T_ = min((int64_t)total_tokens[0], T_cap);
    if (wid >= T_ * Hq) return;
    const T* a = o + wid * D;
    const T* b = dout + wid * D;
    float s = 0.f;
    for (int d = lane; d < D; d += 32) s += to_f(a[d]) * to_f(b[d]);
    s = warp_sum(s);
    if (lane == 0) delta[wid] = s;
}

// dQ for the rows of one query tile and one head.
template <typename T, int DPL>
__global__ void __launch_bounds__(kWarps * 32)
attn_dq_simt_kernel(const QTile* __restrict__ tiles, const int* __restrict__ counts,
                    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                    const float* __restrict__ lse, const float* __restrict__ delta,
                    const T* __restrict__ dout, T* __restrict__ dq, int Hq, int Hkv, float scale,
                    float scale_log2) {
    constexpr int D = DPL * 32;
    __shared__ float sk[kChunk][D + 1];
    __shared__ float sv[kChunk][D + 1];
    if ((int)blockIdx.x >= counts[0]) return;
    const QTile t = tiles[blockIdx.x];
    const int h = blockIdx.y;
    const int hk = h / (Hq / Hkv);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float qr[kRowsPerWarp][DPL], dor[kRowsPerWarp][DPL], acc[kRowsPerWarp][DPL];
    float lrow[kRowsPerWarp], drow[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int row = warp * kRowsPerWarp + r;
        const int64_t rp = t.q0 + min(row, t.nq - 1);
#pragma unroll
        for (int d = 0; d < DPL; ++d) {
            qr[r][d] = to_f(q[(rp * Hq + h) * D + lane + 32 * d]);
            dor[r][d] = to_f(dout[(rp * Hq + h) * D + lane + 32 * d]);
            acc[r][d] = 0.f;
        }
        lrow[r] = lse[rp * Hq + h] * kLog2e;
        drow[r] = delta[rp * Hq + h];
    }
    const int nkeys = (t.pk1 - t.pk0) + (t.q0 + t.nq - t.ck0);
    for (int j0 = 0; j0 < nkeys; j0 += kChunk) {
        __syncthreads();
        for (int i = threadIdx.x; i < kChunk * D; i += blockDim.x) {
            const int jj = i / D, d = i % D;
            const int j = j0 + jj;
            float kv = 0.f, vv = 0.f;
            if (j < nkeys) {
                const int64_t kp = key_pos(t, j);
                kv = to_f(k[(kp * Hkv + hk) * D + d]);
                vv = to_f(v[(kp * Hkv + hk) * D + d]);
            }
            sk[jj][d] = kv;
            sv[jj][d] = vv;
        }
        __syncthreads();
        const int jn = min(kChunk, nkeys - j0);
        for (int jj = 0; jj < jn; ++jj) {
            const int j = j0 + jj;
            const int kp = key_pos(t, j);
            const bool prefix = j < (t.pk1 - t.pk0);
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                const int row = warp * kRowsPerWarp + r;
                if (!(prefix || kp <= t.q0 + row)) continue;
                float s = 0.f, dp = 0.f;
#pragma unroll
                for (int d = 0; d < DPL; ++d) {
                    s += qr[r][d] * sk[jj][lane + 32 * d];
                    dp += dor[r][d] * sv[jj][lane + 32 * d];
                }
                s = warp_sum(s);
                dp = warp_sum(dp);
                const float p = exp2f(s * scale_log2 - lrow[r]);
                const float ds = p * (dp - drow[r]);
#pragma unroll
                for (int d = 0; d < DPL; ++d) acc[r][d] += ds * sk[jj][lane + 32 * d];
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int row = warp * kRowsPerWarp + r;
        if (row >= t.nq) continue;
        const int64_t rp = t.q0 + row;
#pragma unroll
        for (int d = 0; d < DPL; ++d) dq[(rp * Hq + h) * D + lane + 32 * d] = from_f<T>(acc[r][d] * scale);
    }
}

// dK, dV for the keys of one key tile and one key/value head.  The query rows
// that see the tile form contiguous ranges.  Prompt keys (kind 0): prompt rows
// from the tile start to the end of the prompt (causal), then every valid
// response row of the group.  Response keys (kind 1): rows of the same
// response from the tile start (causal).
template <typename T, int DPL>
__global__ void __launch_bounds__(kWarps * 32)
attn_dkdv_simt_kernel(const KTile* __restrict__ tiles, const int* __restrict__ counts,
                      const zr_recon_info info, const T* __restrict__ q, const T* __restrict__ k,
                      const T* __restrict__ v, const float* __restrict__ lse,
                      const float* __restrict__ delta, const T* __restrict__ dout,
                      T* __restrict__ dk, T* __restrict__ dv, int Hq, int Hkv, float scale,
                      float scale_log2) {
    constexpr int D = DPL * 32;
    __shared__ float sq[kChunk][D + 1];
    __shared__ float sdo[kChunk][D + 1];
    __shared__ float sl[kChunk], sd[kChunk];
    __shared__ int spos[kChunk];
    if ((int)blockIdx.x >= counts[1]) return;
    const KTile t = tiles[blockIdx.x];
    const int hk = blockIdx.y;
    const int r_heads = Hq / Hkv;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float kr[kRowsPerWarp][DPL], vr[kRowsPerWarp][DPL], gk[kRowsPerWarp][DPL], gv[kRowsPerWarp][DPL];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int row = warp * kRowsPerWarp + r;
        const int64_t kp = t.k0 + min(row, t.nk - 1);
#pragma unroll
        for (int d = 0; d < DPL; ++d) {
            kr[r][d] = to_f(k[(kp * Hkv + hk) * D + lane + 32 * d]);
            vr[r][d] = to_f(v[(kp * Hkv + hk) * D + lane + 32 * d]);
            gk[r][d] = 0.f;
            gv[r][d] = 0.f;
        }
    }
    // ranges of query rows
    int nrange;
    int rlo[2], rhi[2];
    int m0 = 0, m1 = 0;
    if (t.kind == 0) {
        nrange = 1;
        rlo[0] = t.k0;
        rhi[0] = t.pk1;
        m0 = info.group_ptr[t.g];
        m1 = info.group_ptr[t.g + 1];
    } else {
        nrange = 1;
        rlo[0] = t.k0;
        rhi[0] = info.resp_off[t.b] + info.resp_len[t.b];
    }
    const int nseg = nrange + (m1 - m0);
    for (int hh = 0; hh < r_heads; ++hh) {
        const int h = hk * r_heads + hh;
        for (int sgi = 0; sgi < nseg; ++sgi) {
            int lo, hi;
            bool causal;
            if (sgi < nrange) {
                lo = rlo[sgi]; hi = rhi[sgi]; causal = true;
            } else {
                const int b = info.members[m0 + sgi - nrange];
                lo = info.resp_off[b];
                hi = lo + info.resp_len[b];
                causal = false;
            }
            for (int i0 = lo; i0 < hi; i0 += kChunk) {
                __syncthreads();
                for (int i = threadIdx.x; i < kChunk * D; i += blockDim.x) {
                    const int ii = i / D, d = i % D;
                    const int64_t rp = i0 + ii;
                    float qv = 0.f, dv_ = 0.f;
                    if (rp < hi) {
                        qv = to_f(q[(rp * Hq + h) * D + d]);
                        dv_ = to_f(dout[(rp * Hq + h) * D + d]);
                    }
                    sq[ii][d] = qv;
                    sdo[ii][d] = dv_;
                }
                if (threadIdx.x < kChunk) {
                    const int64_t rp = i0 + threadIdx.x;
                    sl[threadIdx.x] = rp < hi ? lse[rp * Hq + h] * kLog2e : 0.f;
                    sd[threadIdx.x] = rp < hi ? delta[rp * Hq + h] : 0.f;
                    spos[threadIdx.x] = (int)rp;
                }
                __syncthreads();
                const int in_ = min(kChunk, hi - i0);
                for (int ii = 0; ii < in_; ++ii) {
                    const int rp = spos[ii];
#pragma unroll
                    for (int r = 0; r < kRowsPerWarp; ++r) {
                        const int row = warp * kRowsPerWarp + r;
                        if (row >= t.nk) continue;
                        const int kp = t.k0 + row;
                        if (causal && kp > rp) continue;
                        float s = 0.f, dp = 0.f;
#pragma unroll
                        for (int d = 0; d < DPL; ++d) {
                            s += sq[ii][lane + 32 * d] * kr[r][d];
                            dp += sdo[ii][lane + 32 * d] * vr[r][d];
                        }
                        s = warp_sum(s);
                        dp = warp_sum(dp);
                        const float p = exp2f(s * scale_log2 - sl[ii]);
                        const float ds = p * (dp - sd[ii]);
#pragma unroll
                        for (int d = 0; d < DPL; ++d) {
                            gv[r][d] += p * sdo[ii][lane + 32 * d];
                            gk[r][d] += ds * sq[ii][lane + 32 * d];
                        }
                    }
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int row = warp * kRowsPerWarp + r;
        if (row >= t.nk) continue;
        const int64_t kp = t.k0 + row;
#pragma unroll
        for (int d = 0; d < DPL; ++d) {
            dk[(kp * Hkv + hk) * D + lane + 32 * d] = from_f<T>(gk[r][d] * scale);
            dv[(kp * Hkv + hk) * D + lane + 32 * d] = from_f<T>(gv[r][d]);
        }
    }
}

template <typename T, int DPL>
zr_status fwd_dispatch(const AttnWorkspace& ws, const AttnArgs& a, cudaStream_t s) {
    const float scale_log2 = a.scale * kLog2e;
    dim3 grid(ws.plan.max_qtiles, a.Hq);
    attn_fwd_simt_kernel<T, DPL><<<grid, kWarps * 32, 0, s>>>(
        ws.plan.qtiles, ws.plan.counts, static_cast<const T*>(a.q), static_cast<const T*>(a.k),
        static_cast<const T*>(a.v), static_cast<T*>(a.o), a.lse, a.Hq, a.Hkv, scale_log2);
    ZR_LAUNCH_CHECK("attn_fwd_simt_kernel");
    return ZR_OK;
}

template <typename T, int DPL>
zr_status bwd_dispatch(const zr_recon_info& info, const AttnWorkspace& ws, const AttnArgs& a,
                       cudaStream_t s) {
    const float scale_log2 = a.scale * kLog2e;
    dim3 gq(ws.plan.max_qtiles, a.Hq);
    attn_dq_simt_kernel<T, DPL><<<gq, kWarps * 32, 0, s>>>(
        ws.plan.qtiles, ws.plan.counts, static_cast<const T*>(a.q), static_cast<const T*>(a.k),
        static_cast<const T*>(a.v), a.lse_in, ws.delta, static_cast<const T*>(a.dout),
        static_cast<T*>(a.dq), a.Hq, a.Hkv, a.scale, scale_log2);
    ZR_LAUNCH_CHECK("attn_dq_simt_kernel");
    dim3 gk(ws.plan.max_ktiles, a.Hkv);
    attn_dkdv_simt_kernel<T, DPL><<<gk, kWarps * 32, 0, s>>>(
        ws.plan.ktiles, ws.plan.counts, info, static_cast<const T*>(a.q),
        static_cast<const T*>(a.k), static_cast<const T*>(a.v), a.lse_in, ws.delta,
        static_cast<const T*>(a.dout), static_cast<T*>(a.dk), static_cast<T*>(a.dv), a.Hq, a.Hkv,
        a.scale, scale_log2);
    ZR_LAUNCH_CHECK("attn_dkdv_simt_kernel");
    return ZR_OK;
}

template <typename T>
zr_status fwd_by_dim(const AttnWorkspace& ws, const AttnArgs& a, cudaStream_t s) {
    switch (a.D) {
        case 32: return fwd_dispatch<T, 1>(ws, a, s);
        case 64: return fwd_dispatch<T, 2>(ws, a, s);
        case 96: return fwd_dispatch<T, 3>(ws, a, s);
        case 128: return fwd_dispatch<T, 4>(ws, a, s);
        default: return set_error(ZR_ERR_UNSUPPORTED, "SIMT attention: head_dim %d", a.D);
    }
}

template <typename T>
zr_status bwd_by_dim(const zr_recon_info& info, const AttnWorkspace& ws, const AttnArgs& a,
                     cudaStream_t s) {
    switch (a.D) {
        case 32: return bwd_dispatch<T, 1>(info, ws, a, s);
        case 64: return bwd_dispatch<T, 2>(info, ws, a, s);
        case 96: return bwd_dispatch<T, 3>(info, ws, a, s);
        case 128: return bwd_dispatch<T, 4>(info, ws, a, s);
        default: return set_error(ZR_ERR_UNSUPPORTED, "SIMT attention: head_dim %d", a.D);
    }
}

}  // namespace

zr_status launch_attn_fwd_simt(const zr_recon_info& /*info*/, const AttnWorkspace& ws,
                               const AttnArgs& a, cudaStream_t s) {
    if (a.dtype != ZR_F32) return set_error(ZR_ERR_UNSUPPORTED, "SIMT attention is float32 only");
    return fwd_by_dim<float>(ws, a, s);
}

zr_status launch_attn_delta(const zr_recon_info& info, const AttnWorkspace& ws, const AttnArgs& a,
                            cudaStream_t s) {
    const int64_t warps = a.T_cap * a.Hq;
    const int64_t blocks = (warps * 32 + 255) / 256;
    if (a.dtype != ZR_F32) return set_error(ZR_ERR_UNSUPPORTED, "SIMT attention is float32 only");
    attn_delta_kernel<float><<<(unsigned)blocks, 256, 0, s>>>(
        static_cast<const float*>(a.o_in), static_cast<const float*>(a.dout), info.total_tokens,
        a.T_cap, a.Hq, a.D, ws.delta);
    ZR_LAUNCH_CHECK("attn_delta_kernel");
    return ZR_OK;
}

zr_status launch_attn_bwd_simt(const zr_recon_info& info, const AttnWorkspace& ws,
                               const AttnArgs& a, cudaStream_t s) {
    if (a.dtype != ZR_F32) return set_error(ZR_ERR_UNSUPPORTED, "SIMT attention is float32 only");
    return bwd_by_dim<float>(info, ws, a, s);
}

}  // namespace zr
