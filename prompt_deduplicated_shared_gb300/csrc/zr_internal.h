// Internal declarations shared by the translation units of libzr.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "zr.h"

namespace zr {

// ---------------------------------------------------------------- errors
zr_status set_error(zr_status s, const char* fmt, ...);
zr_status cuda_error(cudaError_t e, const char* what);

#define ZR_CUDA_TRY(expr)                                   \
    do {                                                    \
        cudaError_t e_ = (expr);                            \
        if (e_ != cudaSuccess) return zr::cuda_error(e_, #expr); \
    } while (0)

void count_launch();

// An NVTX range named after the entry point, open for the duration of the
// call (profilers show each zr_* call on the host timeline; without a tool
// attached the push and pop cost a few nanoseconds).
class NvtxRange {
public:
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
#define ZR_NVTX(name) ::zr::NvtxRange zr_nvtx_range_(name)

#define ZR_LAUNCH_CHECK(what)                               \
    do {                                                    \
        zr::count_launch();                                 \
        cudaError_t e_ = cudaGetLastError();                \
        if (e_ != cudaSuccess) return zr::cuda_error(e_, what); \
    } while (0)

// Optional per-kernel timing: while the "kernel_timing" option is on, a
// KernelTimer records a CUDA event pair on the launch stream around one launch,
// filed under a short kernel name; zr_kernel_time sums the pairs by name.
class KernelTimer {
public:
    KernelTimer(const char* name, cudaStream_t s);
    ~KernelTimer();
    KernelTimer(const KernelTimer&) = delete;
    KernelTimer& operator=(const KernelTimer&) = delete;
private:
    int slot_ = -1;
    cudaStream_t s_ = nullptr;
};

// process-wide options (zr_set_option)
struct Options {
    int weak_hash = 0;
    int64_t wait_limit = 0;
    int kernel_timing = 0;
    int test_withhold = 0;   // bit 0: forward, bit 1: backward (test option)
};
Options& options();

// device status word slots (zr_recon_info.status / attention workspace)
enum StatusSlot { kStatusMask = 0, kStatusCapacity = 1, kStatusTimeout = 2, kStatusBounds = 3 };

// Debug bounds checks (library built with -DZR_DEBUG_BOUNDS, libzr_debug.so):
// ZR_BOUNDS(cond, status_words, site) is `cond` and, when it fails, records
// `site` in status word kStatusBounds (first failure wins); the caller skips
// the access.  In the normal build it is the constant true.
#ifdef ZR_DEBUG_BOUNDS
#ifdef __CUDACC__
__device__ __forceinline__ bool zr_bounds_ok(bool ok, int32_t* status_words, int site) {
    if (!ok) atomicCAS(status_words + kStatusBounds, 0, site);
    return ok;
}
#endif
#define ZR_BOUNDS(cond, status_words, site) (::zr::zr_bounds_ok((cond), (status_words), (site)))
#else
#define ZR_BOUNDS(cond, status_words, site) true
#endif

// ------------------------------------------------------------- grouping
size_t group_workspace_bytes(int B, int L);
zr_status launch_find_groups(const int64_t* ids, const uint8_t* mask, int B, int L, int P,
                             const zr_groups& out, int64_t* unique_prompts, void* ws,
                             cudaStream_t s);

// --------------------------------------------------------- pack / recon
zr_status launch_pack_plan(const zr_groups& g, const uint8_t* mask, const zr_recon_info& info,
                           cudaStream_t s);
zr_status launch_pack_gather(const zr_recon_info& info, const void* src, int64_t row_bytes,
                             void* dst, cudaStream_t s);
zr_status launch_reconstruct(const zr_recon_info& info, const void* packed, int64_t row_bytes,
                             void* out, cudaStream_t s);
zr_status launch_reconstruct_backward(const zr_recon_info& info, const void* grad_out, int64_t W,
                                      zr_dtype dtype, void* grad_packed, cudaStream_t s);
zr_status launch_pack_backward(const zr_recon_info& info, const void* grad_packed, int64_t row_bytes,
                               void* grad_src, cudaStream_t s);
zr_status launch_reconstruct_pack_backward(const zr_recon_info& info, const void* grad_out, int64_t W,
                                           zr_dtype dtype, void* grad_in, cudaStream_t s);
zr_status launch_batch_stats(const uint8_t* mask, int B, int L, int P, int32_t* plen, int32_t* rlen,
                             int32_t* status, zr_batch_stats* dev_out, cudaStream_t s);
// zero the pad rows (padded mode) of a [T_cap, row_bytes] packed tensor
zr_status launch_zero_pad_rows(const zr_recon_info& info, void* packed, int64_t row_bytes,
                               cudaStream_t s);

// ------------------------------------------------------------ attention
constexpr int kTileM = 128;   // query rows per tile
constexpr int kTileN = 128;   // keys per block

// One query tile: rows [q0, q0+nq) of one prompt or response segment.
// Row r attends [pk0, pk1) (the group's prompt, for response tiles) and the
// causal range [ck0, r].
struct QTile {
    int q0, nq;
    int pk0, pk1;
    int ck0;
    int g;       // group
    int nblk;    // key blocks the tile visits (cost)
    int pad;
};

// One key/value tile: keys [k0, k0+nk) of one segment, for the backward.
// kind 0: prompt keys of group g; kind 1: response keys of sample b.
struct KTile {
    int k0, nk;
    int g, b;
    int kind;
    int nqblk;   // query tiles that see it (cost)
    int pk0, pk1;  // the group's valid prompt rows
};

struct AttnPlan {
    QTile* qtiles;       // [max_qtiles]
    KTile* ktiles;       // [max_ktiles]
    int* counts;         // [8]: 0 n_qtiles, 1 n_ktiles, 2.. scheduler counters
    int* group_qtile_off;  // [B+1] first q tile of each group (q tiles are group-major)
    int* group_ktile_off;  // [B+1]
    // every response query block of group g, in member order, at
    // rblocks[group_ktile_off[g] + i] as (first row, rows)
    int2* rblocks;         // [max_ktiles]
    int max_qtiles, max_ktiles;
};

// rows per head of the backward's (LSE, Delta) pairs: T_cap rounded up to a
// multiple of 4, so that a head's rows start 32-byte aligned (a TMA row stride
// must be a multiple of 16 bytes)
inline int64_t lse_delta_pitch(int64_t T_cap) { return (T_cap + 3) & ~(int64_t)3; }

struct AttnWorkspace {
    AttnPlan plan;
    int* status;         // [4] device status words
    float* delta;        // [T_cap, Hq] rowsum(dO * O), backward only (SIMT)
    // [Hq, lse_delta_pitch(T_cap)] pairs (-LSE * log2(e), rowsum(dO * O)),
    // backward only (tensor cores)
    float2* lse_delta;
    // fp32 dQ accumulator of the tensor-core backward, [Hq, pitch / 4, D, 4]:
    // four consecutive queries interleaved per head-dimension element
    // (pitch = lse_delta_pitch(T_cap))
    float* dq_accum;
    size_t bytes;
};

size_t attn_workspace_layout(const zr_recon_info& info, int Hq, int D, void* base,
                             AttnWorkspace* ws);
zr_status launch_attn_plan(const zr_recon_info& info, const AttnWorkspace& ws, cudaStream_t s);

struct AttnArgs {
    const void* q; const void* k; const void* v;
    void* o; float* lse;
    const void* o_in; const float* lse_in; const void* dout;
    void* dq; void* dk; void* dv;
    int Hq, Hkv, D;
    zr_dtype dtype;
    float scale;
    int64_t T_cap;
};

zr_status launch_attn_fwd_simt(const zr_recon_info& info, const AttnWorkspace& ws,
                               const AttnArgs& a, cudaStream_t s);
zr_status launch_attn_bwd_simt(const zr_recon_info& info, const AttnWorkspace& ws,
                               const AttnArgs& a, cudaStream_t s);
bool tc_fwd_supported(const AttnArgs& a);
bool tc_bwd_supported(const AttnArgs& a);
zr_status launch_attn_fwd_tc(const zr_recon_info& info, const AttnWorkspace& ws,
                             const AttnArgs& a, cudaStream_t s);
zr_status launch_attn_bwd_tc(const zr_recon_info& info, const AttnWorkspace& ws,
                             const AttnArgs& a, cudaStream_t s);
// rowsum(dO * O) per (row, head) for valid rows
zr_status launch_attn_delta(const zr_recon_info& info, const AttnWorkspace& ws,
                            const AttnArgs& a, cudaStream_t s);
// zero LSE of pad rows ([T_cap, Hq] float32)
int num_sms();

}  // namespace zr
