// Work lists of the split-attention kernels, built on the device from the
// reconstruction info so that no host synchronisation is needed.
//
// Query tiles ("Split Attention Optimization"): every valid prompt is cut
// into 128-row tiles that attend causally inside the prompt
// ("Prompt-to-Prompt"); every valid response into 128-row tiles that attend
// the whole valid prompt of their group and causally inside the response
// ("Response-to-Full").  Key tiles cut the same segments for the backward.
//
// Tiles are group-major.  Inside a group they are emitted in descending cost
// (key blocks visited), which is the longest-processing-time-first order for
// the persistent kernels without a sort: every response tile of a group costs
// more than every prompt tile (it scans the whole prompt first), and inside
// each kind the cost grows with the tile index.
#include <cuda_runtime.h>
#include <stdint.h>

#include "zr_internal.h"

namespace zr {
namespace {

constexpr int kMaxPlanGroups = 8192;

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

__device__ int scan_groups(int* data, int n) {
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

__global__ void attn_plan_kernel(zr_recon_info in, AttnPlan plan) {
    extern __shared__ int s_tiles[];  // [B] tiles per group (scanned in place)
    const int B = in.B;
    const int G = in.num_groups[0];
    // nothing to do for an empty batch, or when the packing did not fit T_cap
    const bool empty = in.total_tokens[0] <= 0 || in.total_tokens[0] > in.T_cap;
    for (int g = threadIdx.x; g < B; g += blockDim.x) {
        int n = 0;
        if (g < G && !empty) {
            n = cdiv(in.prompt_len[g], kTileM);
            for (int i = in.group_ptr[g]; i < in.group_ptr[g + 1]; ++i)
                n += cdiv(in.resp_len[in.members[i]], kTileM);
        }
        s_tiles[g] = n;
    }
    __syncthreads();
    const int total = scan_groups(s_tiles, B);
    for (int g = threadIdx.x; g < B; g += blockDim.x) {
        plan.group_qtile_off[g] = s_tiles[g];
        plan.group_ktile_off[g] = s_tiles[g];
    }
    if (threadIdx.x == 0) {
        plan.group_qtile_off[B] = total;
        plan.group_ktile_off[B] = total;
        plan.counts[0] = total;  // query tiles
        plan.counts[1] = total;  // key tiles (same segments)
        for (int i = 2; i < 8; ++i) plan.counts[i] = 0;
    }
    for (int g = threadIdx.x; g < G && !empty; g += blockDim.x) {
        const int plen = in.prompt_len[g];
        const int pv0 = in.prompt_off[g] + in.prompt_slot[g] - plen;
        const int pv1 = pv0 + plen;
        const int npt = cdiv(plen, kTileM);
        const int m0 = in.group_ptr[g], m1 = in.group_ptr[g + 1];
        int max_nrt = 0, sum_nrt = 0;
        for (int i = m0; i < m1; ++i) {
            const int nrt = cdiv(in.resp_len[in.members[i]], kTileM);
            max_nrt = max(max_nrt, nrt);
            sum_nrt += nrt;
        }
        // query tiles, descending cost
        int w = s_tiles[g];
        for (int it = max_nrt - 1; it >= 0; --it) {
            for (int i = m0; i < m1; ++i) {
                const int b = in.members[i];
                const int rlen = in.resp_len[b];
                if (cdiv(rlen, kTileM) <= it) continue;
                QTile t;
                t.q0 = in.resp_off[b] + it * kTileM;
                t.nq = min(kTileM, rlen - it * kTileM);
                t.pk0 = pv0; t.pk1 = pv1;
                t.ck0 = in.resp_off[b];
                t.g = g;
                t.nblk = cdiv(plen, kTileN) + it + 1;
                t.pad = b;
                plan.qtiles[w++] = t;
            }
        }
        for (int it = npt - 1; it >= 0; --it) {
            QTile t;
            t.q0 = pv0 + it * kTileM;
            t.nq = min(kTileM, plen - it * kTileM);
            t.pk0 = 0; t.pk1 = 0;
            t.ck0 = pv0;
            t.g = g;
            t.nblk = it + 1;
            t.pad = -1;
            plan.qtiles[w++] = t;
        }
        // key tiles, descending cost: prompt tiles first, then response tiles
        w = s_tiles[g];
        for (int jt = 0; jt < npt; ++jt) {
            KTile t;
            t.k0 = pv0 + jt * kTileN;
            t.nk = min(kTileN, plen - jt * kTileN);
            t.g = g; t.b = -1; t.kind = 0;
            t.nqblk = (npt - jt) + sum_nrt;
            t.pk0 = pv0; t.pk1 = pv1;
            plan.ktiles[w++] = t;
        }
        // the group's response query blocks in member order (for the backward)
        {
            int wr = s_tiles[g];
            for (int i = m0; i < m1; ++i) {
                const int b = in.members[i];
                const int rlen = in.resp_len[b];
                for (int it = 0; it * kTileM < rlen; ++it)
                    plan.rblocks[wr++] = make_int2(in.resp_off[b] + it * kTileM, min(kTileM, rlen - it * kTileM));
            }
        }
        for (int jt = 0; jt < max_nrt; ++jt) {
            for (int i = m0; i < m1; ++i) {
                const int b = in.members[i];
                const int rlen = in.resp_len[b];
                const int nrt = cdiv(rlen, kTileN);
                if (nrt <= jt) continue;
                KTile t;
                t.k0 = in.resp_off[b] + jt * kTileN;
                t.nk = min(kTileN, rlen - jt * kTileN);
                t.g = g; t.b = b; t.kind = 1;
                t.nqblk = nrt - jt;
                t.pk0 = pv0; t.pk1 = pv1;
                plan.ktiles[w++] = t;
            }
        }
    }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

size_t attn_workspace_layout(const zr_recon_info& info, int Hq, int D, void* base,
                             AttnWorkspace* ws) {
    const int64_t max_tiles = info.T_cap / kTileM + 2 * (int64_t)info.B + 2;
    size_t off = 0;
    char* p = static_cast<char*>(base);
    auto take = [&](size_t bytes) -> void* {
        void* r = p ? p + off : nullptr;
        off += align256(bytes);
        return r;
    };
    AttnWorkspace w;
    w.plan.max_qtiles = (int)max_tiles;
    w.plan.max_ktiles = (int)max_tiles;
    w.plan.qtiles = static_cast<QTile*>(take(sizeof(QTile) * max_tiles));
    w.plan.ktiles = static_cast<KTile*>(take(sizeof(KTile) * max_tiles));
    w.plan.counts = static_cast<int*>(take(sizeof(int) * 8));
    w.plan.group_qtile_off = static_cast<int*>(take(sizeof(int) * (info.B + 1)));
    w.plan.group_ktile_off = static_cast<int*>(take(sizeof(int) * (info.B + 1)));
    w.plan.rblocks = static_cast<int2*>(take(sizeof(int2) * max_tiles));
    w.status = static_cast<int*>(take(sizeof(int) * 4));
    w.delta = static_cast<float*>(take(sizeof(float) * (size_t)info.T_cap * Hq));
    w.lse_delta = static_cast<float2*>(take(sizeof(float2) * (size_t)lse_delta_pitch(info.T_cap) * Hq));
    // fp32 dQ accumulator of the tensor-core backward, [Hq, T_cap, D]
    w.dq_accum = D > 0 ? static_cast<float*>(take(sizeof(float) * (size_t)lse_delta_pitch(info.T_cap) * Hq * D))
                       : nullptr;
    w.bytes = off;
    if (ws) *ws = w;
    return off;
}

zr_status launch_attn_plan(const zr_recon_info& info, const AttnWorkspace& ws, cudaStream_t s) {
    if (info.B > kMaxPlanGroups) return set_error(ZR_ERR_UNSUPPORTED, "B too large");
    const int smem = info.B * (int)sizeof(int);
    ZR_CUDA_TRY(cudaFuncSetAttribute(attn_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kMaxPlanGroups * (int)sizeof(int)));
    attn_plan_kernel<<<1, 1024, smem, s>>>(info, ws.plan);
    ZR_LAUNCH_CHECK("attn_plan_kernel");
    return ZR_OK;
}

}  // namespace zr
