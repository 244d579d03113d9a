// Split attention forward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// "How Prompt Deduplication Works", "Split Attention Optimization": a query
// tile of a prompt attends its prompt causally (prompt-to-prompt, computed
// once per unique prompt); a query tile of a response attends the group's
// whole valid prompt and then its own response causally (response-to-full).
// The tile lists come from zr_attn_plan.cu.
//
// One persistent CTA per SM processes work units (query tile, pair of query
// heads 2p and 2p + 1).  The two heads of a pair are two 128-row query tiles
// that see exactly the same key positions.  When both heads read the same
// key/value head (an even GQA ratio) every K/V block is loaded once by TMA
// and used by both ("GQA packing"); otherwise (odd ratios, MHA) each head
// slot streams the blocks of its own key/value head.  With an odd number of
// query heads the last pair is (Hq - 1, Hq - 1): slot 1 repeats slot 0's head
// and stores nothing.
//
// Warp roles (576 threads):
//   warp 0      TMA producer: Q tiles, then the K/V blocks of each unit in
//               the order the MMAs consume them (shared: K_0, K_1, V_0, K_2,
//               V_1, ...; per slot: K0_0, K1_0, K0_1, V0_0, K1_1, V1_0, ...)
//               through an NS-slot ring
//   warp 1      MMA issuer for both heads, in pipe order: S_t = Q_t K_j^T into
//               TMEM, then, once the softmax has written P_t(j) back into the
//               S_t columns, O_t += P_t(j) V_j with P taken from TMEM; the next
//               block's S_t is issued right after, so the MMAs of one head
//               overlap the other head's softmax.  The loop runs on the whole
//               warp and the elected lane executes tcgen05.  Allocates and frees
//               TMEM.
//   warps 2-17  four softmax warpgroups, two per head: warpgroup (t, part)
//               owns key columns [64 part, +64) of every query row of head t.
//               The two parts exchange their row maxima through shared memory,
//               run the online softmax in base 2 on their 64 columns, write P
//               (bf16 pairs) over the S columns, rescale their half of the O
//               row in TMEM when the running max grew by more than 2^8 (the
//               stale max keeps the result exact, because O and the row sum
//               share it), and finally exchange their row sums and write O / l
//               and the log-sum-exp.
// TMEM columns: O_0 [0, D), O_1 [D, 2D), S_0 [2D, 2D+128), S_1 [2D+128, 2D+256).
//
// Every mbarrier wait is bounded: a wait that runs out sets a CTA-wide abort
// flag and a status word, every role leaves its loop, and the CTA frees its
// TMEM and exits; the host reports ZR_ERR_TIMEOUT.  The softmax warps take
// each wait's outcome as a warp vote so that the warp-collective TMEM
// accesses stay convergent.
//
// Pad rows of q, k and v must hold finite values: masked keys get probability
// 0, and 0 times a non-finite value in V is not 0 in the P V product.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "zr_internal.h"
#include "zr_sm100.cuh"
#include "zr_tc_common.cuh"

namespace zr {
namespace {

using namespace sm100;
using namespace tc;

template <int D>
struct FwdCfg {
    static constexpr int kChunks = D / 64;
    static constexpr int kQBytes = 128 * D * 2;
    static constexpr int kKVBytes = 128 * D * 2;
    static constexpr int kStages = D == 128 ? 4 : 8;
    // qfull, qempty, kvfull[S], kvempty[S], sfull[2], pfull[2], odone[2], xchg[2], unit ring (4), mma drain
    static constexpr int kNumBars = 2 + 2 * kStages + 8 + 4 + 1;
    // row-max exchange [2 parities][2 heads][2 parts][128] and row-sum exchange [2][2][128]
    static constexpr int kXFloats = 2 * 2 * 2 * 128 + 2 * 2 * 128;
    static constexpr int kDataBytes = 2 * kQBytes + kStages * kKVBytes;
    static constexpr int kSmemBytes = kDataBytes + kXFloats * 4 + kNumBars * 8 + 64 + 1024;
    static constexpr uint32_t kColO0 = 0, kColO1 = D, kColS0 = 2 * D, kColS1 = 2 * D + 128;
};

constexpr int kFwdThreads = 576;

struct FwdParams {
    const QTile* qtiles;
    const int* counts;
    const int* group_off;
    int B;
    int npairs;       // query-head pairs, (Hq + 1) / 2
    int ratio;        // Hq / Hkv
    int Hq;
    __nv_bfloat16* o;
    float* lse;
    int64_t T_cap;
    float scale_log2;
    int* status;
    int* sched;       // global unit counter (zeroed by the plan kernel)
    long long limit;
    int withhold;     // test option: the Q load of unit 0 is skipped
};

// Query heads of pair hp (slot 1 repeats the last head when Hq is odd) and
// whether the two slots read different key/value heads.
struct PairHeads {
    int h[2];
    int hk[2];
    bool split;
};
__device__ __forceinline__ PairHeads pair_heads(int hp, int Hq, int ratio) {
    PairHeads r;
    r.h[0] = 2 * hp;
    r.h[1] = min(2 * hp + 1, Hq - 1);
    r.hk[0] = r.h[0] / ratio;
    r.hk[1] = r.h[1] / ratio;
    r.split = r.hk[0] != r.hk[1];
    return r;
}

// Ring position (relative to the unit's first load) of the K/V loads of one
// unit with n key blocks.  W = 1 when the slots share their K/V, else 2 and
// slot t's loads follow slot (t - 1)'s.  Block 0: K_t(0) at t.  Block j in
// [1, n): K_t(j) at W + 2W(j - 1) + 2t and V_t(j - 1) right after it.  Last:
// V_t(n - 1) at W + 2W(n - 1) + t.  A unit takes 2Wn positions.
__device__ __forceinline__ int pos_k(int W, int j, int t) {
    return j == 0 ? t : W + 2 * W * (j - 1) + 2 * t;
}
__device__ __forceinline__ int pos_v(int W, int n, int j, int t) {
    return j == n - 1 ? W + 2 * W * (n - 1) + t : W + 2 * W * j + 2 * t + 1;
}

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s0 = smem_u32(smem);
    const uint32_t sQ0 = s0, sQ1 = s0 + C::kQBytes;
    const uint32_t sKV = s0 + 2 * C::kQBytes;
    float* xmax = reinterpret_cast<float*>(smem + C::kDataBytes);  // [par][t][part][128]
    float* xsum = xmax + 2 * 2 * 2 * 128;                          // [t][part][128]
    const uint32_t bar0 = s0 + C::kDataBytes + C::kXFloats * 4;
    const uint32_t b_qfull = bar0, b_qempty = bar0 + 8;
    auto b_kvfull = [&](int s) { return bar0 + 16 + 8 * s; };
    auto b_kvempty = [&](int s) { return bar0 + 16 + 8 * (C::kStages + s); };
    const uint32_t b_rest = bar0 + 16 + 16 * C::kStages;
    auto b_sfull = [&](int t) { return b_rest + 8 * t; };
    auto b_pfull = [&](int t) { return b_rest + 16 + 8 * t; };
    auto b_odone = [&](int t) { return b_rest + 32 + 8 * t; };
    auto b_xchg = [&](int t) { return b_rest + 48 + 8 * t; };
    uint8_t* misc = smem + C::kDataBytes + C::kXFloats * 4 + C::kNumBars * 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 8);
    const UnitRing ring{b_rest + 64, b_rest + 80, reinterpret_cast<volatile int*>(misc + 16)};
    const uint32_t b_drain = b_rest + 96;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(b_drain, 1);
        mbar_init(b_qfull, 1);
        mbar_init(b_qempty, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(b_kvfull(s), 1);
            mbar_init(b_kvempty(s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(b_sfull(t), 1);
            mbar_init(b_pfull(t), 8);  // one arrival per softmax warp of head t
            mbar_init(b_odone(t), 1);
            mbar_init(b_xchg(t), 8);
        }
        ring_init(ring, 17);  // the MMA warp and 16 softmax warps
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
    const int n_units = p.counts[0] * p.npairs;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            int kstage = 0, k = 0, last_q = -1;
            bool ok = true;
            for (; ok; ++k) {
                const int u = ring_publish(ring, k, p.sched, n_units, ab);
                if (u < 0) { ok = (u == -1); break; }
                int ti, hp;
                decode_unit(u, p.group_off, p.B, p.npairs, ti, hp);
                const QTile t = p.qtiles[ti];
                const PairHeads ph = pair_heads(hp, p.Hq, p.ratio);
                const int W = ph.split ? 2 : 1;
                if (k > 0 && !mbar_wait(b_qempty, (k - 1) & 1, ab, 1)) { ok = false; break; }
                // test option: the CTA that takes unit 0 withholds its Q load, so
                // that a bounded wait runs out and the abort path runs
                if (!(p.withhold && u == 0)) {
                    mbar_expect_tx(b_qfull, 2 * C::kQBytes);
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c) {
                        tma_load_2d(sQ0 + c * kChunkBytes, &tm_q, ph.h[0] * D + 64 * c, t.q0, b_qfull);
                        tma_load_2d(sQ1 + c * kChunkBytes, &tm_q, ph.h[1] * D + 64 * c, t.q0, b_qfull);
                    }
                    last_q = k;
                }
                const int npb = cdiv128(t.pk1 - t.pk0);
                const int n = t.nblk;
                auto load = [&](const CUtensorMap* m, int hk, int row) -> bool {
                    const int slot = kstage % C::kStages, r = kstage / C::kStages;
                    if (r > 0 && !mbar_wait(b_kvempty(slot), (r - 1) & 1, ab, 2)) return false;
                    mbar_expect_tx(b_kvfull(slot), C::kKVBytes);
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_2d(sKV + slot * C::kKVBytes + c * kChunkBytes, m, hk * D + 64 * c, row,
                                    b_kvfull(slot));
                    ++kstage;
                    return true;
                };
                // the order of pos_k / pos_v
                auto hk_of = [&](int w) { return w ? ph.hk[1] : ph.hk[0]; };
                for (int w = 0; w < W && ok; ++w) ok = load(&tm_k, hk_of(w), key_block_row(t, npb, 0));
                for (int j = 1; j < n && ok; ++j)
                    for (int w = 0; w < W && ok; ++w) {
                        ok = load(&tm_k, hk_of(w), key_block_row(t, npb, j));
                        if (ok) ok = load(&tm_v, hk_of(w), key_block_row(t, npb, j - 1));
                    }
                for (int w = 0; w < W && ok; ++w) ok = load(&tm_v, hk_of(w), key_block_row(t, npb, n - 1));
                if (!ok) break;
            }
            const long long lim = p.limit;
            if (ok) {
                // every load consumed and every release committed before exit
                for (int s = kstage - C::kStages; s < kstage; ++s)
                    if (s >= 0) mbar_wait_drain(b_kvempty(s % C::kStages), (s / C::kStages) & 1, lim);
                if (k > 0) mbar_wait_drain(b_qempty, (k - 1) & 1, lim);
            } else {
                // abort: the consumers have left; wait until the copies in flight landed
                for (int s = kstage - C::kStages; s < kstage; ++s)
                    if (s >= 0) mbar_wait_drain(b_kvfull(s % C::kStages), (s / C::kStages) & 1, lim);
                if (last_q >= 0) mbar_wait_drain(b_qfull, last_q & 1, lim);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        const bool leader = elect_one_sync();
        auto wait = [&](uint32_t bar, uint32_t parity, int where) {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, ab, where));
        };
        constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
        // per-slot addresses as selects (a runtime-indexed array would live in
        // local memory on the issue path)
        auto colS = [&](int t) -> uint32_t { return t ? C::kColS1 : C::kColS0; };
        auto colO = [&](int t) -> uint32_t { return t ? C::kColO1 : C::kColO0; };
        auto sQ = [&](int t) -> uint32_t { return t ? sQ1 : sQ0; };
        int base = 0, k = 0;
        int pcnt[2] = {0, 0};
        bool ok = true;
        auto wait_stage = [&](int st) -> int {
            const int slot = st % C::kStages;
            if (!wait(b_kvfull(slot), (st / C::kStages) & 1, 3)) return -1;
            tc_fence_after();
            return slot;
        };
        // S_t = Q_t K^T (K in ring slot kslot)
        auto issue_s = [&](int t, int kslot) {
            const uint64_t dq0 = smem_desc(sQ(t), 16, 1024), dk0 = smem_desc(sKV + kslot * C::kKVBytes, 16, 1024);
#pragma unroll
            for (int s = 0; s < D / 16; ++s) {
                const uint32_t off = ((s >> 2) * kChunkBytes + (s & 3) * 32) >> 4;
                if (leader) mma_bf16_ss(tmem + colS(t), dq0 + off, dk0 + off, idesc_s, s > 0 ? 1u : 0u);
            }
            if (leader) mma_commit(b_sfull(t));
        };
        // O_t (+)= P_t V once the softmax wrote P_t (bf16 pairs in the S_t columns)
        auto issue_pv = [&](int t, int vslot, bool acc) -> bool {
            if (!wait(b_pfull(t), pcnt[t] & 1, 5)) return false;
            ++pcnt[t];
            tc_fence_after();
            const uint64_t dv0 = smem_desc(sKV + vslot * C::kKVBytes, kChunkBytes, 1024);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                if (leader)
                    mma_bf16_ts(tmem + colO(t), tmem + colS(t) + 8 * s, dv0 + s * 128, idesc_pv,
                                (acc || s > 0) ? 1u : 0u);
            return true;
        };
        for (; ok; ++k) {
            const int u = ring_take_warp(ring, k, ab);
            if (u < 0) { ok = (u == -1); break; }
            int ti, hp;
            decode_unit(u, p.group_off, p.B, p.npairs, ti, hp);
            const int n = p.qtiles[ti].nblk;
            const int W = pair_heads(hp, p.Hq, p.ratio).split ? 2 : 1;
            if (!wait(b_qfull, k & 1, 6)) { ok = false; break; }
            tc_fence_after();
            // ring positions from pos_k / pos_v; slot t reads the loads of w = t
            // when the slots stream their own K/V (W = 2), else those of w = 0.
            // A stage is released once its last reader was issued: after slot t
            // (W = 2) or after slot 1 (W = 1).
            for (int t = 0; t < 2 && ok; ++t) {
                const int w = W == 2 ? t : 0;
                int kslot = (t == 0 || W == 2) ? wait_stage(base + pos_k(W, 0, w)) : -2;
                if (kslot == -1) { ok = false; break; }
                if (kslot == -2) kslot = (base + pos_k(W, 0, 0)) % C::kStages;
                issue_s(t, kslot);
                if (leader && (W == 2 || t == 1)) mma_commit(b_kvempty(kslot));
            }
            if (!ok) break;
            if (n == 1 && leader) mma_commit(b_qempty);
            for (int j = 1; j < n && ok; ++j) {
                for (int t = 0; t < 2; ++t) {
                    const int w = W == 2 ? t : 0;
                    const int kst = base + pos_k(W, j, w), vst = base + pos_v(W, n, j - 1, w);
                    int kslot, vslot;
                    if (t == 0 || W == 2) {
                        kslot = wait_stage(kst);
                        vslot = kslot < 0 ? -1 : wait_stage(vst);
                        if (vslot < 0) { ok = false; break; }
                    } else {
                        kslot = kst % C::kStages;
                        vslot = vst % C::kStages;
                    }
                    if (!issue_pv(t, vslot, j > 1)) { ok = false; break; }
                    issue_s(t, kslot);
                    if (leader && (W == 2 || t == 1)) {
                        mma_commit(b_kvempty(vslot));
                        mma_commit(b_kvempty(kslot));
                    }
                }
                if (!ok) break;
                if (leader && j == n - 1) mma_commit(b_qempty);
            }
            if (!ok) break;
            for (int t = 0; t < 2 && ok; ++t) {
                const int w = W == 2 ? t : 0;
                const int vst = base + pos_v(W, n, n - 1, w);
                int vslot = (t == 0 || W == 2) ? wait_stage(vst) : vst % C::kStages;
                if (vslot < 0) { ok = false; break; }
                if (!issue_pv(t, vslot, n > 1)) { ok = false; break; }
                if (leader) mma_commit(b_odone(t));
                if (leader && (W == 2 || t == 1)) mma_commit(b_kvempty(vslot));
            }
            if (!ok) break;
            base += 2 * W * n;
        }
        drain_mmas(leader, b_drain, p.limit);
    } else {
        // ------------------------------------------------------ softmax
        const int wg = (warp - 2) >> 2;
        const int t = wg >> 1, part = wg & 1;  // head t, key columns [64 part, +64)
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t colS = t ? C::kColS1 : C::kColS0;
        const uint32_t colO = (t ? C::kColO1 : C::kColO0) + (D / 2) * part;  // this part's half of O
        const float sl2 = p.scale_log2;
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        int s_cnt = 0, x_cnt = 0, o_cnt = 0;
        bool ok = true;
        // one arrival per warp, after every lane's shared-memory write
        auto xwait = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(b_xchg(t));
            const bool w = __all_sync(0xffffffffu, mbar_wait(b_xchg(t), x_cnt & 1, ab, 10));
            ++x_cnt;
            return w;
        };
        for (int k = 0; ok; ++k) {
            const int u = ring_take_warp(ring, k, ab);
            if (u < 0) { ok = (u == -1); break; }
            int ti, hp;
            decode_unit(u, p.group_off, p.B, p.npairs, ti, hp);
            const QTile tile = p.qtiles[ti];
            const PairHeads ph = pair_heads(hp, p.Hq, p.ratio);
            const int h = t ? ph.h[1] : ph.h[0];
            // slot 1 of the last pair of an odd head count repeats slot 0's head
            const bool own_head = t == 0 || 2 * hp + 1 < p.Hq;
            const int npb = cdiv128(tile.pk1 - tile.pk0);
            const int n = tile.nblk;
            const int row_pos = tile.q0 + r;
            float m = -1e30f, l = 0.f;
            for (int j = 0; j < n; ++j) {
                if (!__all_sync(0xffffffffu, mbar_wait(b_sfull(t), s_cnt & 1, ab, 7))) { ok = false; break; }
                ++s_cnt;
                tc_fence_after();
                uint32_t sr[2][32];
                tmem_ld32(trow + colS + 64 * part, sr[0]);
                tmem_ld32(trow + colS + 64 * part + 32, sr[1]);
                tmem_wait_ld();
                const int kbase = key_block_row(tile, npb, j);
                const int lim = (j < npb ? (tile.pk1 - kbase) : (row_pos - kbase + 1)) - 64 * part;
                if (lim < 64) {
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (32 * c + i >= lim) sr[c][i] = __float_as_uint(-INFINITY);
                }
                // partial row max as 8 independent chains, then the exchange
                float mxv[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) mxv[q] = -INFINITY;
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) mxv[i & 7] = fmaxf(mxv[i & 7], __uint_as_float(sr[c][i]));
                const float mxp = fmaxf(fmaxf(fmaxf(mxv[0], mxv[1]), fmaxf(mxv[2], mxv[3])),
                                        fmaxf(fmaxf(mxv[4], mxv[5]), fmaxf(mxv[6], mxv[7])));
                float* xm = xmax + (((x_cnt & 1) * 2 + t) * 2) * 128;
                xm[part * 128 + r] = mxp;
                if (!xwait()) { ok = false; break; }
                const float mx = fmaxf(mxp, xm[(1 - part) * 128 + r]);
                const float mnew = fmaxf(m, mx * sl2);
                // rescale when the running max grew by more than 2^8 (j > 0); the O
                // rescale itself waits until the S registers are dead
                const bool need = j > 0 && mnew > m + 8.0f;
                const float alpha = need ? ex2(m - mnew) : 1.0f;
                if (j == 0 || need) m = mnew;
                const uint64_t mneg2 = f2_pack(-m, -m);
                // row sum as 8 independent partial sums, held as four fp32 pairs;
                // exponent arguments and sums two columns per instruction
                uint64_t lp2[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) lp2[q] = 0ull;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1])), sl2x2,
                                         mneg2),
                                  x0, x1);
                        const float e0 = ex2(x0);
                        const float e1 = ex2(x1);
                        lp2[(i & 7) >> 1] = f2_add(lp2[(i & 7) >> 1], f2_pack(e0, e1));
                        pk[i >> 1] = pack_bf16x2(e0, e1);
                    }
                    // P (bf16 pairs) of keys [64 part + 32 c, +32) over S columns already read
                    tmem_st16(trow + colS + 32 * part + 16 * c, pk);
                }
                float lp[8];
#pragma unroll
                for (int q = 0; q < 4; ++q) f2_unpack(lp2[q], lp[2 * q], lp[2 * q + 1]);
                l = l * alpha + (((lp[0] + lp[1]) + (lp[2] + lp[3])) + ((lp[4] + lp[5]) + (lp[6] + lp[7])));
                // O_t holds P V up to block j - 1: its last MMA completed before S_t(j),
                // whose completion this thread observed; P V of block j waits for pfull
                if (__any_sync(0xffffffffu, need)) {
                    const uint64_t alpha2 = f2_pack(alpha, alpha);
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {
                        uint32_t o[32];
                        tmem_ld32(trow + colO + 32 * c, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            float a0, a1;
                            f2_unpack(f2_mul(f2_pack(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), alpha2), a0, a1);
                            o[i] = __float_as_uint(a0);
                            o[i + 1] = __float_as_uint(a1);
                        }
                        tmem_st32(trow + colO + 32 * c, o);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(b_pfull(t));
            }
            if (!ok) break;
            // epilogue: row sums exchanged, O / l for this part's half, the log-sum-exp
            if (!__all_sync(0xffffffffu, mbar_wait(b_odone(t), o_cnt & 1, ab, 9))) { ok = false; break; }
            ++o_cnt;
            tc_fence_after();
            float* xs = xsum + t * 2 * 128;
            xs[part * 128 + r] = l;
            if (!xwait()) { ok = false; break; }
            const float ltot = l + xs[(1 - part) * 128 + r];
            const float inv = 1.0f / ltot;
            const bool store =
                r < tile.nq && own_head && ZR_BOUNDS(row_pos < p.T_cap, p.status - kStatusTimeout, 10);
            __nv_bfloat16* orow = p.o + ((int64_t)row_pos * p.Hq + h) * D + (D / 2) * part;
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t o[32];
                tmem_ld32(trow + colO + 32 * c, o);
                tmem_wait_ld();
                if (store) {
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(o[i + 0]) * inv, __uint_as_float(o[i + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(o[i + 4]) * inv, __uint_as_float(o[i + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(o[i + 6]) * inv, __uint_as_float(o[i + 7]) * inv);
                        *reinterpret_cast<uint4*>(orow + 32 * c + i) = w;
                    }
                }
            }
            if (store && part == 0) p.lse[(int64_t)row_pos * p.Hq + h] = (m + __log2f(ltot)) * kLn2;
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
zr_status launch_fwd(const zr_recon_info& info, const AttnWorkspace& ws, const AttnArgs& a, cudaStream_t s) {
    using C = FwdCfg<D>;
    CUtensorMap tq, tk, tv;
    zr_status st;
    if ((st = make_map(&tq, a.q, (int64_t)a.Hq * D, a.T_cap, (int64_t)a.Hq * D * 2)) != ZR_OK) return st;
    if ((st = make_map(&tk, a.k, (int64_t)a.Hkv * D, a.T_cap, (int64_t)a.Hkv * D * 2)) != ZR_OK) return st;
    if ((st = make_map(&tv, a.v, (int64_t)a.Hkv * D, a.T_cap, (int64_t)a.Hkv * D * 2)) != ZR_OK) return st;
    FwdParams p;
    p.qtiles = ws.plan.qtiles;
    p.counts = ws.plan.counts;
    p.group_off = ws.plan.group_qtile_off;
    p.B = info.B;
    p.npairs = (a.Hq + 1) / 2;
    p.ratio = a.Hq / a.Hkv;
    p.Hq = a.Hq;
    p.o = static_cast<__nv_bfloat16*>(a.o);
    p.lse = a.lse;
    p.T_cap = a.T_cap;
    p.scale_log2 = a.scale * kLog2e;
    p.status = info.status + kStatusTimeout;  // read by zr_check_status(info)
    p.sched = ws.plan.counts + 2;
    p.limit = wait_limit_cycles();
    p.withhold = (options().test_withhold & 1) != 0;
    ZR_CUDA_TRY(cudaFuncSetAttribute(attn_fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::kSmemBytes));
    {
        KernelTimer timer("attn_fwd", s);
        attn_fwd_tc_kernel<D><<<num_sms(), kFwdThreads, C::kSmemBytes, s>>>(tq, tk, tv, p);
        ZR_LAUNCH_CHECK("attn_fwd_tc_kernel");
    }
    return ZR_OK;
}

}  // namespace

bool tc_fwd_supported(const AttnArgs& a) {
    return a.dtype == ZR_BF16 && (a.D == 64 || a.D == 128) && a.Hkv > 0 && a.Hq % a.Hkv == 0;
}

zr_status launch_attn_fwd_tc(const zr_recon_info& info, const AttnWorkspace& ws, const AttnArgs& a,
                             cudaStream_t s) {
    if (a.D == 128) return launch_fwd<128>(info, ws, a, s);
    return launch_fwd<64>(info, ws, a, s);
}

}  // namespace zr
