// Split attention backward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// "How Prompt Deduplication Works", "Correctness & Gradients": gradients flow
// through the deduplicated attention; a prompt key's dK and dV collect the
// contributions of the prompt's own queries and of every response of its
// group.  The probabilities are recomputed from the forward's log-sum-exp:
// P = 2^(S * scale * log2(e) - LSE * log2(e)), dS = P * (dP - Delta) with
// Delta = rowsum(dO * O), dV = P^T dO, dK = scale * dS^T Q, dQ = scale * dS K.
//
// Three launches:
//   attn_bwd_prep_kernel  Delta and LSE (base 2) per (head, row), head-major
//   attn_dq_tc_kernel     query-tile-major: per work unit (query tile, head)
//                         Q and dO sit in TMEM and the key blocks stream
//                         through a three-stage TMA ring; S = Q K^T and
//                         dP = dO V^T go to TMEM; four softmax warpgroups (32
//                         key columns each) form dS in shared memory; dQ += dS K
//                         accumulates in TMEM.
//   attn_dkdv_tc_kernel   key-tile-major: per work unit (key tile, key/value
//                         head) the K and V tiles stay in shared memory while
//                         the query blocks that see them (all query heads of
//                         the group) stream through a TMA ring; S^T = K Q^T and
//                         dP^T = V dO^T go to TMEM; four softmax warpgroups (32
//                         query columns each) write P^T back to TMEM (bf16) and
//                         dS^T to shared memory; dV += P^T dO takes its A
//                         operand from TMEM, dK += dS^T Q from shared memory.
// The query blocks that see a prompt key tile are the prompt's own blocks
// from the diagonal on (causal) and every block of every response of the
// group; a response key tile is seen by its own response's blocks from the
// diagonal on.
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

// Delta = rowsum(dO * O) and LSE * log2(e), head-major [Hq, T_cap], rows < T.
__global__ void attn_bwd_prep_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                                     const float* __restrict__ lse, const int32_t* __restrict__ total_tokens,
                                     int64_t T_cap, int Hq, int D, float* __restrict__ delta_t,
                                     float* __restrict__ lse2_t) {
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
    // reduce over the row's lanes (groups of G consecutive lanes, G a power of two)
    for (int off = G >> 1; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (valid && part == 0) {
        const int64_t t = row / Hq;
        const int h = (int)(row - t * Hq);
        delta_t[(int64_t)h * T_cap + t] = s;
        lse2_t[(int64_t)h * T_cap + t] = lse[row] * kLog2e;
    }
}

struct BwdParams {
    const QTile* qtiles;
    const KTile* ktiles;
    const int* counts;
    const int* qgroup_off;
    const int* kgroup_off;
    const int32_t* group_ptr;
    const int32_t* members;
    const int32_t* resp_off;
    const int32_t* resp_len;
    const int2* rblocks;
    const __nv_bfloat16* q;
    const __nv_bfloat16* dout;
    int B;
    int Hq, Hkv, ratio;
    const float* delta_t;
    const float* lse2_t;
    int64_t T_cap;
    __nv_bfloat16* dq;
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    float scale;
    float scale_log2;
    int* status;
    int* sched;       // global unit counters (zeroed by the plan kernel): [0] dK/dV, [1] dQ
    long long limit;
};

// ======================================================================= dQ
// Q and dO of the unit's query tile live in TMEM (written by the softmax
// warpgroups from global memory), so the S = Q K^T and dP = dO V^T GEMMs take
// their A operand from TMEM and shared memory holds three K/V stages.
template <int D>
struct DqCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kTile = 128 * D * 2;  // one K or V block
    static constexpr int kStages = D == 128 ? 3 : 6;
    // kvfull[S], kvempty[S], qd_ready, sdp_full, sdp_free, ds_full, mm_done, unit ring (4), mma drain
    static constexpr int kNumBars = 2 * kStages + 5 + 4 + 1;
    static constexpr int kDS = 128 * 128 * 2;
    static constexpr int kDataBytes = kStages * 2 * kTile + kDS;
    static constexpr int kSmemBytes = kDataBytes + kNumBars * 8 + 64 + 1024;
    // TMEM: S [0, 128), dP [128, 256), dQ [256, 256 + D), Q [256 + D, +D/2), dO [256 + 3D/2, +D/2)
    static constexpr uint32_t kColS = 0, kColP = 128, kColQ = 256;
    static constexpr uint32_t kColQin = 256 + D, kColDO = 256 + D + D / 2;
};

constexpr int kDqThreads = 640;  // producer, MMA issuer, 2 idle warps, 4 softmax warpgroups

template <int D>
__global__ void __launch_bounds__(kDqThreads, 1)
attn_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const BwdParams p) {
    using C = DqCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s0 = smem_u32(smem);
    const uint32_t sKV = s0;  // stage s: K at sKV + s*2*kTile, V at + kTile
    const uint32_t sDS = sKV + C::kStages * 2 * C::kTile;
    const uint32_t bar0 = s0 + C::kDataBytes;
    auto b_kvfull = [&](int s) { return bar0 + 8 * s; };
    auto b_kvempty = [&](int s) { return bar0 + 8 * (C::kStages + s); };
    const uint32_t b_rest = bar0 + 16 * C::kStages;
    const uint32_t b_qdready = b_rest, b_sdpfull = b_rest + 8, b_sdpfree = b_rest + 16, b_dsfull = b_rest + 24,
                   b_mmdone = b_rest + 32;
    uint8_t* misc = smem + C::kDataBytes + C::kNumBars * 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 8);
    const UnitRing ring{b_rest + 40, b_rest + 56, reinterpret_cast<volatile int*>(misc + 16)};
    const uint32_t b_drain = b_rest + 72;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(b_drain, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(b_kvfull(s), 1);
            mbar_init(b_kvempty(s), 1);
        }
        mbar_init(b_qdready, 512);
        mbar_init(b_sdpfull, 1);
        mbar_init(b_sdpfree, 512);
        mbar_init(b_dsfull, 512);
        mbar_init(b_mmdone, 1);
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
    const int n_units = p.counts[0] * p.Hq;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            int kstage = 0, k = 0;
            bool ok = true;
            for (; ok; ++k) {
                const int u = ring_publish(ring, k, p.sched + 1, n_units, ab);
                if (u < 0) { ok = (u == -1); break; }
                int ti, h;
                decode_unit(u, p.qgroup_off, p.B, p.Hq, ti, h);
                const QTile t = p.qtiles[ti];
                const int hk = h / p.ratio;
                const int npb = cdiv128(t.pk1 - t.pk0);
                for (int j = 0; j < t.nblk; ++j) {
                    const int slot = kstage % C::kStages, r = kstage / C::kStages;
                    if (r > 0 && !mbar_wait(b_kvempty(slot), (r - 1) & 1, ab, 22)) { ok = false; break; }
                    mbar_expect_tx(b_kvfull(slot), 2 * C::kTile);
                    const int row = key_block_row(t, npb, j);
                    const uint32_t kb = sKV + slot * 2 * C::kTile;
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c) {
                        tma_load_2d(kb + c * kChunkBytes, &tm_k, hk * D + 64 * c, row, b_kvfull(slot));
                        tma_load_2d(kb + C::kTile + c * kChunkBytes, &tm_v, hk * D + 64 * c, row, b_kvfull(slot));
                    }
                    ++kstage;
                }
            }
            const long long lim = p.limit;
            for (int s = kstage - C::kStages; s < kstage; ++s)
                if (s >= 0) mbar_wait_drain(b_kvempty(s % C::kStages), (s / C::kStages) & 1, lim);
        }
    } else if (warp == 1) {
        // the whole warp runs the issue loop (warp-uniform state); the elected
        // lane executes the tcgen05 instructions
        {
            const bool leader = elect_one_sync();
            auto wait = [&](uint32_t bar, uint32_t parity, int where) {
                return __all_sync(0xffffffffu, mbar_wait(bar, parity, ab, where));
            };
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
            constexpr uint32_t idesc_dq = idesc_bf16_f32(128, D, false, true);
            int kstage = 0, k = 0, sdp_cnt = 0, ds_cnt = 0;
            bool ok = true;
            for (; ok; ++k) {
                const int u = ring_take_warp(ring, k, ab);
                if (u < 0) { ok = (u == -1); break; }
                int ti, h;
                decode_unit(u, p.qgroup_off, p.B, p.Hq, ti, h);
                const int n = p.qtiles[ti].nblk;
                if (!wait(b_qdready, k & 1, 23)) { ok = false; break; }
                tc_fence_after();
                int prev_slot = -1;
                for (int j = 0; j <= n && ok; ++j) {
                    int slot = -1;
                    if (j < n) {
                        slot = kstage % C::kStages;
                        if (!wait(b_kvfull(slot), (kstage / C::kStages) & 1, 24)) { ok = false; break; }
                        ++kstage;
                        // S / dP TMEM free: the softmax has read the previous pair
                        if (sdp_cnt > 0 && !wait(b_sdpfree, (sdp_cnt - 1) & 1, 25)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t kb = sKV + slot * 2 * C::kTile;
                        const uint64_t dk0 = smem_desc(kb, 16, 1024), dv0 = smem_desc(kb + C::kTile, 16, 1024);
#pragma unroll
                        for (int s = 0; s < D / 16; ++s) {
                            const uint32_t off = ((s >> 2) * kChunkBytes + (s & 3) * 32) >> 4;
                            if (leader) mma_bf16_ts(tmem + C::kColS, tmem + C::kColQin + 8 * s, dk0 + off, idesc_s,
                                                    s > 0 ? 1u : 0u);
                        }
#pragma unroll
                        for (int s = 0; s < D / 16; ++s) {
                            const uint32_t off = ((s >> 2) * kChunkBytes + (s & 3) * 32) >> 4;
                            if (leader) mma_bf16_ts(tmem + C::kColP, tmem + C::kColDO + 8 * s, dv0 + off, idesc_s,
                                                    s > 0 ? 1u : 0u);
                        }
                        if (leader) mma_commit(b_sdpfull);
                        ++sdp_cnt;
                    }
                    if (j > 0) {
                        // dQ += dS K for the previous key block
                        if (!wait(b_dsfull, ds_cnt & 1, 26)) { ok = false; break; }
                        ++ds_cnt;
                        tc_fence_after();
                        const uint32_t kb = sKV + prev_slot * 2 * C::kTile;
                        const uint64_t da0 = smem_desc(sDS, 16, 1024), db0 = smem_desc(kb, kChunkBytes, 1024);
#pragma unroll
                        for (int s = 0; s < 8; ++s) {
                            const uint32_t aoff = ((s >> 2) * kChunkBytes + (s & 3) * 32) >> 4;
                            if (leader) mma_bf16_ss(tmem + C::kColQ, da0 + aoff, db0 + s * 128, idesc_dq,
                                                    (j > 1 || s > 0) ? 1u : 0u);
                        }
                        if (leader) mma_commit(b_mmdone);
                        if (leader) mma_commit(b_kvempty(prev_slot));
                    }
                    prev_slot = slot;
                }
            }
            drain_mmas(leader, b_drain, p.limit);
        }
    } else if (warp >= 4) {
        // Four softmax warpgroups; warpgroup wg owns key columns [32 wg, 32 wg + 32)
        // of S and dP for all 128 query rows (one query row per thread).
        const int wg = (warp - 4) >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t drow = sDS + (wg >> 1) * kChunkBytes + (r >> 3) * 1024 + (r & 7) * 128;
        const int piece0 = (wg & 1) * 4;
        const float sl2 = p.scale_log2;
        int sdp_cnt = 0, mm_cnt = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int u = ring_take_warp(ring, k, ab);
            if (u < 0) { ok = (u == -1); break; }
            int ti, h;
            decode_unit(u, p.qgroup_off, p.B, p.Hq, ti, h);
            const QTile t = p.qtiles[ti];
            const int npb = cdiv128(t.pk1 - t.pk0);
            const int row_pos = t.q0 + r;
            const bool valid_row = r < t.nq;
            // this warpgroup's share of the row's Q and dO (32 head-dim columns; for
            // D = 64 warpgroups 0-1 cover the row) into TMEM as bf16 pairs
            if (D == 128 || wg < 2) {
                uint32_t qv[16], dv[16];
                if (row_pos < p.T_cap) {
                    const uint4* qs = reinterpret_cast<const uint4*>(p.q + ((int64_t)row_pos * p.Hq + h) * D + 32 * wg);
                    const uint4* ds = reinterpret_cast<const uint4*>(p.dout + ((int64_t)row_pos * p.Hq + h) * D + 32 * wg);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint4 a4 = __ldg(qs + i), b4 = __ldg(ds + i);
                        qv[4 * i] = a4.x; qv[4 * i + 1] = a4.y; qv[4 * i + 2] = a4.z; qv[4 * i + 3] = a4.w;
                        dv[4 * i] = b4.x; dv[4 * i + 1] = b4.y; dv[4 * i + 2] = b4.z; dv[4 * i + 3] = b4.w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) { qv[i] = 0u; dv[i] = 0u; }
                }
                tmem_st16(trow + C::kColQin + 16 * wg, qv);
                tmem_st16(trow + C::kColDO + 16 * wg, dv);
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(b_qdready);
            const float lse2 = valid_row ? p.lse2_t[(int64_t)h * p.T_cap + row_pos] : INFINITY;
            const float dlt = valid_row ? p.delta_t[(int64_t)h * p.T_cap + row_pos] : 0.f;
            for (int j = 0; j < t.nblk; ++j) {
                if (!__all_sync(0xffffffffu, mbar_wait(b_sdpfull, sdp_cnt & 1, ab, 27))) { ok = false; break; }
                ++sdp_cnt;
                tc_fence_after();
                uint32_t sr[32], dr[32];
                tmem_ld32(trow + C::kColS + 32 * wg, sr);
                tmem_ld32(trow + C::kColP + 32 * wg, dr);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(b_sdpfree);
                const int kbase = key_block_row(t, npb, j);
                const int lim = (j < npb ? (t.pk1 - kbase) : (row_pos - kbase + 1)) - 32 * wg;
                // dS (bf16 pairs) in registers first; the shared-memory copy waits until
                // the previous dQ MMA has finished reading the dS buffer
                uint32_t dsv[16];
                auto block = [&](auto masked) {
                    constexpr bool kMasked = decltype(masked)::value;
#pragma unroll
                    for (int pc = 0; pc < 4; ++pc) {
                        float v[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int col = 8 * pc + i;
                            float pr = ex2(fmaf(__uint_as_float(sr[col]), sl2, -lse2));
                            if (kMasked) pr = (col < lim) ? pr : 0.f;
                            v[i] = pr * (__uint_as_float(dr[col]) - dlt);
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) dsv[4 * pc + i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
                    }
                };
                if (__any_sync(0xffffffffu, lim < 32)) block(std::integral_constant<bool, true>());
                else block(std::integral_constant<bool, false>());
                if (j > 0) {
                    if (!__all_sync(0xffffffffu, mbar_wait(b_mmdone, mm_cnt & 1, ab, 28))) { ok = false; break; }
                    ++mm_cnt;
                }
#pragma unroll
                for (int pc = 0; pc < 4; ++pc)
                    st_shared_v4_nc(drow + (((piece0 + pc) ^ (r & 7)) << 4), dsv[4 * pc], dsv[4 * pc + 1],
                                    dsv[4 * pc + 2], dsv[4 * pc + 3]);
                fence_async_smem();
                tc_fence_before();
                mbar_arrive(b_dsfull);
            }
            if (!ok) break;
            // epilogue: dQ = scale * accumulated dS K; warpgroup wg writes columns
            // [wg D/4, (wg+1) D/4)
            if (!__all_sync(0xffffffffu, mbar_wait(b_mmdone, mm_cnt & 1, ab, 29))) { ok = false; break; }
            ++mm_cnt;
            tc_fence_after();
            __nv_bfloat16* out = p.dq + ((int64_t)row_pos * p.Hq + h) * D + wg * (D / 4);
            if constexpr (D == 128) {
                uint32_t o[32];
                tmem_ld32(trow + C::kColQ + wg * 32, o);
                tmem_wait_ld();
                if (valid_row) {
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(o[i + 0]) * p.scale, __uint_as_float(o[i + 1]) * p.scale);
                        w.y = pack_bf16x2(__uint_as_float(o[i + 2]) * p.scale, __uint_as_float(o[i + 3]) * p.scale);
                        w.z = pack_bf16x2(__uint_as_float(o[i + 4]) * p.scale, __uint_as_float(o[i + 5]) * p.scale);
                        w.w = pack_bf16x2(__uint_as_float(o[i + 6]) * p.scale, __uint_as_float(o[i + 7]) * p.scale);
                        *reinterpret_cast<uint4*>(out + i) = w;
                    }
                }
            } else {
                uint32_t o[16];
                tmem_ld16(trow + C::kColQ + wg * 16, o);
                tmem_wait_ld();
                if (valid_row) {
#pragma unroll
                    for (int i = 0; i < 16; i += 8) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(o[i + 0]) * p.scale, __uint_as_float(o[i + 1]) * p.scale);
                        w.y = pack_bf16x2(__uint_as_float(o[i + 2]) * p.scale, __uint_as_float(o[i + 3]) * p.scale);
                        w.z = pack_bf16x2(__uint_as_float(o[i + 4]) * p.scale, __uint_as_float(o[i + 5]) * p.scale);
                        w.w = pack_bf16x2(__uint_as_float(o[i + 6]) * p.scale, __uint_as_float(o[i + 7]) * p.scale);
                        *reinterpret_cast<uint4*>(out + i) = w;
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

// =================================================================== dK, dV
template <int D>
struct DkvCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kTile = 128 * D * 2;
    // Q and dO are staged per 64-query half: a half-slot holds Q_h then dO_h,
    // each kChunks chunks of 64 rows x 64 columns (8 KB, 128-byte swizzle)
    static constexpr int kHalfChunk = 64 * 128;
    static constexpr int kHalf = 64 * D * 2;
    static constexpr int kStages = D == 128 ? 4 : 8;  // half-slots
    // kfull, kempty, qfull[S], qempty[S], sdp_full[2], pds_full[2], (2 unused), unit ring (4), mma drain
    static constexpr int kNumBars = 2 + 2 * kStages + 6 + 4 + 1;
    static constexpr int kDataBytes = 2 * kTile + kStages * 2 * kHalf;
    // data, LSE/Delta staging (2 KB), barriers, misc words, alignment slack
    static constexpr int kSmemBytes = kDataBytes + 2048 + kNumBars * 8 + 64 + 1024;
    // TMEM: dV [0, D), dK [D, 2D); query half h: S^T [2D + 128h, +64), dP^T [2D + 128h + 64, +64);
    // the softmax writes P^T and dS^T (bf16 pairs) back over the first half of
    // the S^T and dP^T columns it read
    static constexpr uint32_t kColV = 0, kColK = D;
    __host__ __device__ static constexpr uint32_t col_s(int h) { return 2 * D + 128 * h; }
    __host__ __device__ static constexpr uint32_t col_p(int h) { return 2 * D + 128 * h + 64; }
};

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
constexpr int kDkvThreads = 576;

// Each 128-query block is processed as two 64-query halves A and B with their
// own S^T / dP^T columns in TMEM, so that one half's softmax overlaps the
// other half's GEMMs.  MMA order per block `it`:
//   S^T_A, dP^T_A (it) | dV, dK += half B (it-1) | S^T_B, dP^T_B (it) | dV, dK += half A (it)
// The four softmax warpgroups take half A, then half B, 16 query columns each
// (warpgroup g: columns [16 g, +16) of the half); a warpgroup writes its P^T
// and dS^T (bf16 pairs) over the first 8 of the 16 S^T and dP^T columns it
// read, which is exactly the A operand of K step g of the accumulations, so no
// other warpgroup's values are overwritten.  Both accumulations take their A operand from TMEM, so shared
// memory only feeds K, V, Q and dO to the tensor cores.  The next block's
// S^T / dP^T GEMMs of a half are issued after that half's accumulations, and
// MMAs of one thread complete in order, so TMEM reuse needs no extra wait.
template <int D>
__global__ void __launch_bounds__(kDkvThreads, 1)
attn_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BwdParams p) {
    using C = DkvCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s0 = smem_u32(smem);
    const uint32_t sK = s0, sV = s0 + C::kTile;
    const uint32_t sQD = s0 + 2 * C::kTile;  // half-slot s: Q_h at sQD + s*2*kHalf, dO_h at + kHalf
    float* stage_f = reinterpret_cast<float*>(smem + C::kDataBytes);  // [16 warps][32]: 16 LSE, 16 Delta
    const uint32_t bar0 = s0 + C::kDataBytes + 2048;
    const uint32_t b_kfull = bar0, b_kempty = bar0 + 8;
    auto b_qfull = [&](int s) { return bar0 + 16 + 8 * s; };
    auto b_qempty = [&](int s) { return bar0 + 16 + 8 * (C::kStages + s); };
    const uint32_t b_rest = bar0 + 16 + 16 * C::kStages;
    auto b_sdpfull = [&](int h) { return b_rest + 8 * h; };
    auto b_pdsfull = [&](int h) { return b_rest + 16 + 8 * h; };
    uint8_t* misc = smem + C::kDataBytes + 2048 + C::kNumBars * 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 8);
    const UnitRing ring{b_rest + 48, b_rest + 64, reinterpret_cast<volatile int*>(misc + 16)};
    const uint32_t b_drain = b_rest + 80;

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
            mbar_init(b_sdpfull(h), 1);
            mbar_init(b_pdsfull(h), 512);
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
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_do);
            int qstage = 0, k = 0;
            bool ok = true;
            for (; ok; ++k) {
                const int u = ring_publish(ring, k, p.sched, n_units, ab);
                if (u < 0) { ok = (u == -1); break; }
                int ti, hk;
                decode_unit(u, p.kgroup_off, p.B, p.Hkv, ti, hk);
                const KTile t = p.ktiles[ti];
                if (k > 0 && !mbar_wait(b_kempty, (k - 1) & 1, ab, 31)) { ok = false; break; }
                mbar_expect_tx(b_kfull, 2 * C::kTile);
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_2d(sK + c * kChunkBytes, &tm_k, hk * D + 64 * c, t.k0, b_kfull);
                    tma_load_2d(sV + c * kChunkBytes, &tm_v, hk * D + 64 * c, t.k0, b_kfull);
                }
                const int rb_base = t.kind == 0 ? p.kgroup_off[t.g] : 0;
                for (int hh = 0; hh < p.ratio && ok; ++hh) {
                    const int h = hk * p.ratio + hh;
                    for (int qi = 0; qi < t.nqblk && ok; ++qi) {
                        const QBlock qb = qblock_of(t, p, qi, rb_base);
                        for (int half = 0; half < 2; ++half) {
                            const int slot = qstage % C::kStages, r = qstage / C::kStages;
                            if (r > 0 && !mbar_wait(b_qempty(slot), (r - 1) & 1, ab, 32)) { ok = false; break; }
                            mbar_expect_tx(b_qfull(slot), 2 * C::kHalf);
                            const uint32_t qb_s = sQD + slot * 2 * C::kHalf;
                            const int row = qb.q0 + 64 * half;
#pragma unroll
                            for (int c = 0; c < C::kChunks; ++c) {
                                tma_load_2d(qb_s + c * C::kHalfChunk, &tm_q, h * D + 64 * c, row, b_qfull(slot));
                                tma_load_2d(qb_s + C::kHalf + c * C::kHalfChunk, &tm_do, h * D + 64 * c, row,
                                            b_qfull(slot));
                            }
                            ++qstage;
                        }
                    }
                }
            }
            const long long lim = p.limit;
            for (int s = qstage - C::kStages; s < qstage; ++s)
                if (s >= 0) mbar_wait_drain(b_qempty(s % C::kStages), (s / C::kStages) & 1, lim);
            if (k > 0) mbar_wait_drain(b_kempty, (k - 1) & 1, lim);
        }
    } else if (warp == 1) {
        // the whole warp runs the issue loop (warp-uniform state); the elected
        // lane executes the tcgen05 instructions
        {
            const bool leader = elect_one_sync();
            auto wait = [&](uint32_t bar, uint32_t parity, int where) {
                return __all_sync(0xffffffffu, mbar_wait(bar, parity, ab, where));
            };
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, 64, false, false);
            constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, false, true);
            int qstage = 0, k = 0, pds_cnt[2] = {0, 0};
            bool ok = true;
            // base descriptors; a K step adds a compile-time offset (in 16-byte
            // units) to the start-address field, which never carries out of it
            const uint64_t dK0 = smem_desc(sK, 16, 1024), dV0 = smem_desc(sV, 16, 1024);
            // S^T_h = K Q_h^T and dP^T_h = V dO_h^T for query half h (half-slot `slot`)
            auto issue_sdp = [&](int slot, int h) {
                const uint32_t qh = sQD + slot * 2 * C::kHalf, dh = qh + C::kHalf;
                const uint64_t dq0 = smem_desc(qh, 16, 1024), ddo0 = smem_desc(dh, 16, 1024);
#pragma unroll
                for (int s = 0; s < D / 16; ++s) {
                    const uint32_t ka = ((s >> 2) * kChunkBytes + (s & 3) * 32) >> 4;
                    const uint32_t qa = ((s >> 2) * C::kHalfChunk + (s & 3) * 32) >> 4;
                    if (leader) mma_bf16_ss(tmem + C::col_s(h), dK0 + ka, dq0 + qa, idesc_s, s > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int s = 0; s < D / 16; ++s) {
                    const uint32_t ka = ((s >> 2) * kChunkBytes + (s & 3) * 32) >> 4;
                    const uint32_t qa = ((s >> 2) * C::kHalfChunk + (s & 3) * 32) >> 4;
                    if (leader) mma_bf16_ss(tmem + C::col_p(h), dV0 + ka, ddo0 + qa, idesc_s, s > 0 ? 1u : 0u);
                }
                if (leader) mma_commit(b_sdpfull(h));
            };
            // dV += P^T_h dO_h, dK += dS^T_h Q_h (both A operands from TMEM); first = overwrite
            auto issue_acc = [&](int slot, int h, bool first) -> bool {
                if (!wait(b_pdsfull(h), pds_cnt[h] & 1, 35)) return false;
                ++pds_cnt[h];
                tc_fence_after();
                const uint32_t qh = sQD + slot * 2 * C::kHalf, dh = qh + C::kHalf;
                const uint64_t bq0 = smem_desc(qh, C::kHalfChunk, 1024), bdo0 = smem_desc(dh, C::kHalfChunk, 1024);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    if (leader) mma_bf16_ts(tmem + C::kColV, tmem + C::col_s(h) + 16 * s, bdo0 + s * 128, idesc_acc,
                                            (!first || s > 0) ? 1u : 0u);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    if (leader) mma_bf16_ts(tmem + C::kColK, tmem + C::col_p(h) + 16 * s, bq0 + s * 128, idesc_acc,
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
                    issue_sdp(slot_a, 0);
                    if (it > 0) {
                        if (!issue_acc(prev_b, 1, false)) { ok = false; break; }
                        if (leader) mma_commit(b_qempty(prev_b));
                    }
                    const int slot_b = qstage % C::kStages;
                    if (!wait(b_qfull(slot_b), (qstage / C::kStages) & 1, 34)) { ok = false; break; }
                    ++qstage;
                    tc_fence_after();
                    issue_sdp(slot_b, 1);
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
        }
    } else {
        // softmax warps: warpgroup wg owns query columns [16 wg, +16) of each
        // 64-query half; all four warpgroups take half A, then half B
        const int wg = (warp - 2) >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // key row
        const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
        float* st = stage_f + (warp - 2) * 32;  // this warp's 16 LSE (base 2) then 16 Delta
        const float sl2 = p.scale_log2;
        int sdp_cnt[2] = {0, 0};
        bool ok = true;
        // lane < 16: LSE of query column 16 wg + lane of half `hf`; lane >= 16: its Delta
        auto stage_value = [&](const QBlock& qb, int hf, int hh_, int hk_) -> float {
            const int h = hk_ * p.ratio + hh_;
            const int qc = 64 * hf + 16 * wg + (lane & 15);
            if (qc >= qb.nq) return lane < 16 ? INFINITY : 0.f;
            return lane < 16 ? p.lse2_t[(int64_t)h * p.T_cap + qb.q0 + qc]
                             : p.delta_t[(int64_t)h * p.T_cap + qb.q0 + qc];
        };
        for (int k = 0; ok; ++k) {
            const int u = ring_take_warp(ring, k, ab);
            if (u < 0) { ok = (u == -1); break; }
            int ti, hk;
            decode_unit(u, p.kgroup_off, p.B, p.Hkv, ti, hk);
            const KTile t = p.ktiles[ti];
            const int key_pos = t.k0 + r;
            const int iters = t.nqblk * p.ratio;
            const int rb_base = t.kind == 0 ? p.kgroup_off[t.g] : 0;
            QBlock qb_next = qblock_of(t, p, 0, rb_base);
            float pre_next = stage_value(qb_next, 0, 0, hk);
            for (int it = 0; it < iters && ok; ++it) {
                const QBlock qb = qb_next;
                if (it + 1 < iters) qb_next = qblock_of(t, p, (it + 1) % t.nqblk, rb_base);
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const float pre = pre_next;
                    // the value staged for the next half, loaded before this half's
                    // S^T is awaited so that its latency hides behind the wait
                    if (hf == 0) pre_next = stage_value(qb, 1, it / t.nqblk, hk);
                    else if (it + 1 < iters) pre_next = stage_value(qb_next, 0, (it + 1) / t.nqblk, hk);
                    if (!__all_sync(0xffffffffu, mbar_wait(b_sdpfull(hf), sdp_cnt[hf] & 1, ab, 36))) {
                        ok = false;
                        break;
                    }
                    ++sdp_cnt[hf];
                    tc_fence_after();
                    uint32_t sr[16], dr[16];
                    tmem_ld16(trow + C::col_s(hf) + 16 * wg, sr);
                    tmem_ld16(trow + C::col_p(hf) + 16 * wg, dr);
                    st[lane] = pre;
                    __syncwarp();
                    tmem_wait_ld();
                    uint32_t pk[8], dk[8];
                    const int qlo = key_pos - qb.q0 - 64 * hf - 16 * wg;  // causal: query >= key
                    auto block = [&](auto masked) {
                        constexpr bool kMasked = decltype(masked)::value;
#pragma unroll
                        for (int pc = 0; pc < 2; ++pc) {
                            const float4 l0 = *reinterpret_cast<const float4*>(st + 8 * pc);
                            const float4 l1 = *reinterpret_cast<const float4*>(st + 8 * pc + 4);
                            const float4 d0 = *reinterpret_cast<const float4*>(st + 16 + 8 * pc);
                            const float4 d1 = *reinterpret_cast<const float4*>(st + 16 + 8 * pc + 4);
                            const float lv[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
                            const float dv[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
                            float pv[8], ds[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const int col = 8 * pc + i;
                                float pr = ex2(fmaf(__uint_as_float(sr[col]), sl2, -lv[i]));
                                if (kMasked) pr = (col >= qlo) ? pr : 0.f;
                                pv[i] = pr;
                                ds[i] = pr * (__uint_as_float(dr[col]) - dv[i]);
                            }
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                pk[4 * pc + i] = pack_bf16x2(pv[2 * i], pv[2 * i + 1]);
                                dk[4 * pc + i] = pack_bf16x2(ds[2 * i], ds[2 * i + 1]);
                            }
                        }
                    };
                    if (qb.diag) block(std::integral_constant<bool, true>());
                    else block(std::integral_constant<bool, false>());
                    // P^T and dS^T (bf16 pairs) over the first 8 of the 16 columns read
                    tmem_st8(trow + C::col_s(hf) + 16 * wg, pk);
                    tmem_st8(trow + C::col_p(hf) + 16 * wg, dk);
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(b_pdsfull(hf));
                    __syncwarp();  // every lane read `st` before the next half rewrites it
                }
            }
            if (!ok) break;
            // epilogue: every MMA of unit k is done once its kempty phase completed (the
            // MMA thread commits it after the unit's last accumulation; the next unit
            // cannot finish before this epilogue, so the phase parity is unambiguous).
            // Warpgroups 0-1 write dV columns [64 wg, +64), 2-3 write scale * dK.
            if (!__all_sync(0xffffffffu, mbar_wait(b_kempty, k & 1, ab, 38))) { ok = false; break; }
            tc_fence_after();
            const bool store = r < t.nk;
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
    CUtensorMap tq, tk, tv, tdo;
    zr_status st;
    // Q and dO: 64-row boxes (the dK/dV kernel stages them per 64-query half)
    if ((st = make_map(&tq, a.q, (int64_t)a.Hq * D, a.T_cap, (int64_t)a.Hq * D * 2, 64)) != ZR_OK) return st;
    if ((st = make_map(&tdo, a.dout, (int64_t)a.Hq * D, a.T_cap, (int64_t)a.Hq * D * 2, 64)) != ZR_OK) return st;
    if ((st = make_map(&tk, a.k, (int64_t)a.Hkv * D, a.T_cap, (int64_t)a.Hkv * D * 2)) != ZR_OK) return st;
    if ((st = make_map(&tv, a.v, (int64_t)a.Hkv * D, a.T_cap, (int64_t)a.Hkv * D * 2)) != ZR_OK) return st;
    {
        const int64_t threads = a.T_cap * a.Hq * (D / 8);
        const int64_t blocks = (threads + 255) / 256;
        KernelTimer timer("attn_bwd_prep", s);
        attn_bwd_prep_kernel<<<(unsigned)blocks, 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(a.o_in), static_cast<const __nv_bfloat16*>(a.dout), a.lse_in,
            info.total_tokens, a.T_cap, a.Hq, D, ws.delta_t, ws.lse2_t);
        ZR_LAUNCH_CHECK("attn_bwd_prep_kernel");
    }
    BwdParams p;
    p.qtiles = ws.plan.qtiles;
    p.ktiles = ws.plan.ktiles;
    p.counts = ws.plan.counts;
    p.qgroup_off = ws.plan.group_qtile_off;
    p.kgroup_off = ws.plan.group_ktile_off;
    p.group_ptr = info.group_ptr;
    p.members = info.members;
    p.resp_off = info.resp_off;
    p.resp_len = info.resp_len;
    p.rblocks = ws.plan.rblocks;
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.dout = static_cast<const __nv_bfloat16*>(a.dout);
    p.B = info.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.ratio = a.Hq / a.Hkv;
    p.delta_t = ws.delta_t;
    p.lse2_t = ws.lse2_t;
    p.T_cap = a.T_cap;
    p.dq = static_cast<__nv_bfloat16*>(a.dq);
    p.dk = static_cast<__nv_bfloat16*>(a.dk);
    p.dv = static_cast<__nv_bfloat16*>(a.dv);
    p.scale = a.scale;
    p.scale_log2 = a.scale * kLog2e;
    p.status = info.status + kStatusTimeout;  // read by zr_check_status(info)
    p.sched = ws.plan.counts + 3;
    p.limit = wait_limit_cycles();
    ZR_CUDA_TRY(cudaFuncSetAttribute(attn_dkdv_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     DkvCfg<D>::kSmemBytes));
    ZR_CUDA_TRY(cudaFuncSetAttribute(attn_dq_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     DqCfg<D>::kSmemBytes));
    {
        KernelTimer timer("attn_dkdv", s);
        attn_dkdv_tc_kernel<D><<<num_sms(), kDkvThreads, DkvCfg<D>::kSmemBytes, s>>>(tq, tk, tv, tdo, p);
        ZR_LAUNCH_CHECK("attn_dkdv_tc_kernel");
    }
    {
        KernelTimer timer("attn_dq", s);
        attn_dq_tc_kernel<D><<<num_sms(), kDqThreads, DqCfg<D>::kSmemBytes, s>>>(tk, tv, p);
        ZR_LAUNCH_CHECK("attn_dq_tc_kernel");
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
