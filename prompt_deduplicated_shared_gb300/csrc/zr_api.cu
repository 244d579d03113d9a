// extern "C" entry points of libzr: host-side validation, workspace layout and
// launch sequencing.  Every compute step runs in the kernels of the other
// translation units.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "zr_internal.h"

namespace zr {

namespace {
thread_local char g_msg[512] = "no error";
std::atomic<int64_t> g_launches{0};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool aligned256(const void* p) { return ((uintptr_t)p & 255) == 0; }

zr_status check_info(const zr_recon_info* info) {
    if (!info) return set_error(ZR_ERR_INVALID_ARG, "info is NULL");
    if (!info->prompt_off || !info->status || !info->recon_segs || info->B <= 0 || info->L <= 0 ||
        info->P < 0 || info->P > info->L || info->T_cap <= 0)
        return set_error(ZR_ERR_INVALID_ARG, "reconstruction info is not bound");
    return ZR_OK;
}
}  // namespace

zr_status set_error(zr_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return s;
}

zr_status cuda_error(cudaError_t e, const char* what) {
    return set_error(ZR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {
// Event pairs recorded by KernelTimer.  Bounded so that a caller who leaves
// timing on never grows it without limit; pairs past the bound are dropped and
// counted, and zr_kernel_time reports them as an error.
constexpr size_t kMaxTimed = 1 << 14;
struct TimedLaunch {
    std::string name;
    cudaEvent_t start = nullptr, stop = nullptr;
    bool used = false;
};
std::mutex g_timing_mu;
std::vector<TimedLaunch> g_timed;
std::vector<cudaEvent_t> g_event_pool;
int64_t g_timing_dropped = 0;

cudaEvent_t take_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}
}  // namespace

KernelTimer::KernelTimer(const char* name, cudaStream_t s) : s_(s) {
    if (!options().kernel_timing) return;
    std::lock_guard<std::mutex> lk(g_timing_mu);
    if (g_timed.size() >= kMaxTimed) {
        ++g_timing_dropped;
        return;
    }
    TimedLaunch t;
    t.name = name;
    t.start = take_event();
    t.stop = take_event();
    if (!t.start || !t.stop || cudaEventRecord(t.start, s) != cudaSuccess) {
        if (t.start) g_event_pool.push_back(t.start);
        if (t.stop) g_event_pool.push_back(t.stop);
        ++g_timing_dropped;
        return;
    }
    slot_ = (int)g_timed.size();
    g_timed.push_back(t);
}

KernelTimer::~KernelTimer() {
    if (slot_ < 0) return;
    std::lock_guard<std::mutex> lk(g_timing_mu);
    if (slot_ < (int)g_timed.size() && cudaEventRecord(g_timed[slot_].stop, s_) == cudaSuccess)
        g_timed[slot_].used = true;
    else
        ++g_timing_dropped;
}

Options& options() {
    static Options o;
    return o;
}

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
    return n;
}

}  // namespace zr

using namespace zr;

extern "C" {

const char* zr_last_error(void) { return g_msg; }

int zr_version(void) { return 100; }

int zr_debug_bounds(void) {
#ifdef ZR_DEBUG_BOUNDS
    return 1;
#else
    return 0;
#endif
}

int64_t zr_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

zr_status zr_set_option(const char* name, int64_t value) {
    if (!name) return set_error(ZR_ERR_INVALID_ARG, "option name is NULL");
    if (!strcmp(name, "weak_hash")) {
        options().weak_hash = value != 0;
    } else if (!strcmp(name, "wait_limit")) {
        if (value < 0) return set_error(ZR_ERR_INVALID_ARG, "wait_limit must be >= 0");
        options().wait_limit = value;
    } else if (!strcmp(name, "kernel_timing")) {
        options().kernel_timing = value != 0;
    } else if (!strcmp(name, "test_withhold_arrival")) {
        if (value < 0 || value > 3) return set_error(ZR_ERR_INVALID_ARG, "test_withhold_arrival must be 0..3");
        options().test_withhold = (int)value;
    } else {
        return set_error(ZR_ERR_INVALID_ARG, "unknown option '%s'", name);
    }
    return ZR_OK;
}

zr_status zr_kernel_time(const char* name, double* total_ms, int64_t* launches) {
    if (!name || !total_ms || !launches)
        return set_error(ZR_ERR_INVALID_ARG, "NULL name or output of zr_kernel_time");
    std::lock_guard<std::mutex> lk(g_timing_mu);
    double sum = 0.0;
    int64_t n = 0;
    for (const TimedLaunch& t : g_timed) {
        if (!t.used || t.name != name) continue;
        ZR_CUDA_TRY(cudaEventSynchronize(t.stop));
        float ms = 0.f;
        ZR_CUDA_TRY(cudaEventElapsedTime(&ms, t.start, t.stop));
        sum += ms;
        ++n;
    }
    *total_ms = sum;
    *launches = n;
    if (g_timing_dropped)
        return set_error(ZR_ERR_CAPACITY, "%lld timed launches were dropped (more than %zu recorded)",
                         (long long)g_timing_dropped, kMaxTimed);
    return ZR_OK;
}

zr_status zr_kernel_time_reset(void) {
    std::lock_guard<std::mutex> lk(g_timing_mu);
    for (TimedLaunch& t : g_timed) {
        if (t.used) ZR_CUDA_TRY(cudaEventSynchronize(t.stop));
        g_event_pool.push_back(t.start);
        g_event_pool.push_back(t.stop);
    }
    g_timed.clear();
    g_timing_dropped = 0;
    return ZR_OK;
}

size_t zr_find_prompt_groups_workspace(int B, int L) {
    if (B <= 0) return 0;
    return group_workspace_bytes(B, L);
}

zr_status zr_find_prompt_groups(const int64_t* input_ids, const uint8_t* attention_mask, int B,
                                int L, int response_length, const zr_groups* out,
                                int64_t* unique_prompts, int32_t* num_groups_host, void* workspace,
                                size_t workspace_bytes, void* stream) {
    ZR_NVTX("zr_find_prompt_groups");
    if (!input_ids || !out || !out->group_ptr || !out->members || !out->group_of || !out->num_groups)
        return set_error(ZR_ERR_INVALID_ARG, "NULL input_ids or group output");
    if (B <= 0 || L <= 0) return set_error(ZR_ERR_INVALID_ARG, "B and L must be positive (B=%d L=%d)", B, L);
    if (response_length < 0 || response_length > L)
        return set_error(ZR_ERR_INVALID_ARG, "response_length %d outside [0, L=%d]", response_length, L);
    if (B > 8192) return set_error(ZR_ERR_UNSUPPORTED, "B=%d exceeds 8192 rows", B);
    const size_t need = group_workspace_bytes(B, L);
    if (!workspace || workspace_bytes < need || !aligned256(workspace))
        return set_error(ZR_ERR_WORKSPACE, "group workspace needs %zu bytes, 256-aligned", need);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    zr_status st = launch_find_groups(input_ids, attention_mask, B, L, L - response_length, *out,
                                      unique_prompts, workspace, s);
    if (st != ZR_OK) return st;
    if (num_groups_host) {
        ZR_CUDA_TRY(cudaMemcpyAsync(num_groups_host, out->num_groups, sizeof(int32_t),
                                    cudaMemcpyDeviceToHost, s));
        ZR_CUDA_TRY(cudaStreamSynchronize(s));
    }
    return ZR_OK;
}

size_t zr_recon_info_bytes(int B) {
    if (B <= 0) return 0;
    const size_t b4 = align256((size_t)B * 4);
    return 10 * b4 + align256((size_t)(B + 1) * 4) + 2 * align256(16) +
           align256((size_t)2 * B * 24) * 3 + align256((size_t)4 * B * 24);
}

zr_status zr_recon_info_bind(zr_recon_info* info, void* buffer, int B, int L, int response_length,
                             int use_unpad, int64_t T_cap) {
    if (!info || !buffer) return set_error(ZR_ERR_INVALID_ARG, "NULL info or buffer");
    if (!aligned256(buffer)) return set_error(ZR_ERR_INVALID_ARG, "buffer must be 256-byte aligned");
    if (B <= 0 || L <= 0 || response_length < 0 || response_length > L)
        return set_error(ZR_ERR_INVALID_ARG, "bad sizes B=%d L=%d response_length=%d", B, L, response_length);
    if (B > 8192) return set_error(ZR_ERR_UNSUPPORTED, "B=%d exceeds 8192 rows", B);
    if (T_cap <= 0 || T_cap > (int64_t)B * L || T_cap > INT32_MAX)
        return set_error(ZR_ERR_INVALID_ARG, "T_cap %lld outside [1, B*L]", (long long)T_cap);
    char* p = static_cast<char*>(buffer);
    size_t off = 0;
    auto take = [&](size_t bytes) -> void* {
        void* r = p + off;
        off += align256(bytes);
        return r;
    };
    const size_t b4 = (size_t)B * 4;
    info->prompt_off = static_cast<int32_t*>(take(b4));
    info->prompt_slot = static_cast<int32_t*>(take(b4));
    info->prompt_len = static_cast<int32_t*>(take(b4));
    info->resp_off = static_cast<int32_t*>(take(b4));
    info->resp_slot = static_cast<int32_t*>(take(b4));
    info->resp_len = static_cast<int32_t*>(take(b4));
    info->group_ptr = static_cast<int32_t*>(take((size_t)(B + 1) * 4));
    info->members = static_cast<int32_t*>(take(b4));
    info->group_of = static_cast<int32_t*>(take(b4));
    info->num_groups = static_cast<int32_t*>(take(16));
    info->total_tokens = static_cast<int32_t*>(take(16));
    info->status = static_cast<int32_t*>(take(b4 < 16 ? 16 : b4));
    info->row_prompt_len = static_cast<int32_t*>(take(b4));
    info->pack_segs = static_cast<int64_t*>(take((size_t)2 * B * 24));
    info->pad_segs = static_cast<int64_t*>(take((size_t)2 * B * 24));
    info->recon_segs = static_cast<int64_t*>(take((size_t)4 * B * 24));
    info->pack_order = static_cast<int64_t*>(take((size_t)2 * B * 24));
    if (off > zr_recon_info_bytes(B)) return set_error(ZR_ERR_INVALID_ARG, "internal layout error");
    info->B = B;
    info->L = L;
    info->P = L - response_length;
    info->use_unpad = use_unpad ? 1 : 0;
    info->T_cap = T_cap;
    return ZR_OK;
}

zr_status zr_pack_dedup(const int64_t* input_ids, const int64_t* position_ids,
                        const uint8_t* attention_mask, const zr_groups* groups,
                        int64_t* dedup_input_ids, int64_t* dedup_position_ids, uint8_t* dedup_mask,
                        zr_recon_info* info, int64_t* T_host, void* stream) {
    ZR_NVTX("zr_pack_dedup");
    zr_status st = check_info(info);
    if (st != ZR_OK) return st;
    if (!input_ids || !groups || !groups->group_ptr || !groups->members || !groups->group_of ||
        !groups->num_groups || !dedup_input_ids)
        return set_error(ZR_ERR_INVALID_ARG, "NULL input_ids, groups or dedup_input_ids");
    if (position_ids && !dedup_position_ids)
        return set_error(ZR_ERR_INVALID_ARG, "position_ids given without dedup_position_ids");
    if (info->use_unpad && !attention_mask)
        return set_error(ZR_ERR_INVALID_ARG, "use_unpad needs an attention_mask");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = launch_pack_plan(*groups, attention_mask, *info, s);
    if (st != ZR_OK) return st;
    if (T_host) {
        int32_t hv[2];
        int32_t hs[4];
        ZR_CUDA_TRY(cudaMemcpyAsync(hv, info->total_tokens, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
        ZR_CUDA_TRY(cudaMemcpyAsync(hs, info->status, sizeof(hs), cudaMemcpyDeviceToHost, s));
        ZR_CUDA_TRY(cudaStreamSynchronize(s));
        *T_host = hv[0];
        if (hs[kStatusMask]) return set_error(ZR_ERR_INVALID_ARG, "attention_mask layout unsupported: "
                                              "prompts must be left padded and responses right padded");
        if (hs[kStatusCapacity])
            return set_error(ZR_ERR_CAPACITY, "packed tokens %d exceed T_cap %lld", hv[0], (long long)info->T_cap);
    }
    const int64_t B = info->B, L = info->L;
    (void)B; (void)L;
    st = launch_pack_gather(*info, input_ids, 8, dedup_input_ids, s);
    if (st != ZR_OK) return st;
    if (position_ids) {
        st = launch_pack_gather(*info, position_ids, 8, dedup_position_ids, s);
        if (st != ZR_OK) return st;
    }
    if (dedup_mask) {
        if (attention_mask) {
            st = launch_pack_gather(*info, attention_mask, 1, dedup_mask, s);
            if (st != ZR_OK) return st;
        } else {
            ZR_CUDA_TRY(cudaMemsetAsync(dedup_mask, 1, (size_t)info->T_cap, s));
        }
    }
    return ZR_OK;
}

zr_status zr_pack_rows(const zr_recon_info* info, const void* src, int64_t row_bytes, void* dst,
                       void* stream) {
    ZR_NVTX("zr_pack_rows");
    zr_status st = check_info(info);
    if (st != ZR_OK) return st;
    if (!src || !dst || row_bytes <= 0) return set_error(ZR_ERR_INVALID_ARG, "NULL src/dst or row_bytes <= 0");
    return launch_pack_gather(*info, src, row_bytes, dst, static_cast<cudaStream_t>(stream));
}

zr_status zr_reconstruct(const zr_recon_info* info, const void* packed, int64_t row_bytes, void* out,
                         void* stream) {
    ZR_NVTX("zr_reconstruct");
    zr_status st = check_info(info);
    if (st != ZR_OK) return st;
    if (!packed || !out || row_bytes <= 0)
        return set_error(ZR_ERR_INVALID_ARG, "NULL packed/out or row_bytes <= 0");
    return launch_reconstruct(*info, packed, row_bytes, out, static_cast<cudaStream_t>(stream));
}

zr_status zr_reconstruct_backward(const zr_recon_info* info, const void* grad_out, int64_t W, int dtype,
                                  void* grad_packed, void* stream) {
    ZR_NVTX("zr_reconstruct_backward");
    zr_status st = check_info(info);
    if (st != ZR_OK) return st;
    if (!grad_out || !grad_packed || W <= 0)
        return set_error(ZR_ERR_INVALID_ARG, "NULL grad_out/grad_packed or W <= 0");
    if (dtype != ZR_BF16 && dtype != ZR_F32)
        return set_error(ZR_ERR_UNSUPPORTED, "reconstruct_backward supports ZR_BF16 and ZR_F32 elements");
    return launch_reconstruct_backward(*info, grad_out, W, static_cast<zr_dtype>(dtype), grad_packed,
                                       static_cast<cudaStream_t>(stream));
}

zr_status zr_pack_rows_backward(const zr_recon_info* info, const void* grad_packed, int64_t row_bytes,
                                void* grad_src, void* stream) {
    ZR_NVTX("zr_pack_rows_backward");
    zr_status st = check_info(info);
    if (st != ZR_OK) return st;
    if (!grad_packed || !grad_src || row_bytes <= 0)
        return set_error(ZR_ERR_INVALID_ARG, "NULL grad_packed/grad_src or row_bytes <= 0");
    return launch_pack_backward(*info, grad_packed, row_bytes, grad_src, static_cast<cudaStream_t>(stream));
}

zr_status zr_reconstruct_pack_backward(const zr_recon_info* info, const void* grad_out, int64_t W, int dtype,
                                       void* grad_in, void* stream) {
    ZR_NVTX("zr_reconstruct_pack_backward");
    zr_status st = check_info(info);
    if (st != ZR_OK) return st;
    if (!grad_out || !grad_in || W <= 0) return set_error(ZR_ERR_INVALID_ARG, "NULL grad_out/grad_in or W <= 0");
    if (grad_out == grad_in) return set_error(ZR_ERR_INVALID_ARG, "grad_in must not alias grad_out");
    if (dtype != ZR_BF16 && dtype != ZR_F32)
        return set_error(ZR_ERR_UNSUPPORTED, "reconstruct_pack_backward supports ZR_BF16 and ZR_F32 elements");
    return launch_reconstruct_pack_backward(*info, grad_out, W, static_cast<zr_dtype>(dtype), grad_in,
                                            static_cast<cudaStream_t>(stream));
}

size_t zr_batch_stats_workspace(int B) {
    if (B <= 0) return 0;
    return 2 * align256((size_t)B * 4) + align256(16) + align256(sizeof(zr_batch_stats));
}

zr_status zr_batch_stats_compute(const uint8_t* attention_mask, int B, int L, int response_length,
                                 zr_batch_stats* out, void* workspace, size_t workspace_bytes, void* stream) {
    ZR_NVTX("zr_batch_stats_compute");
    if (!out) return set_error(ZR_ERR_INVALID_ARG, "NULL output");
    if (B <= 0 || L <= 0 || response_length < 0 || response_length > L)
        return set_error(ZR_ERR_INVALID_ARG, "bad sizes B=%d L=%d response_length=%d", B, L, response_length);
    const size_t need = zr_batch_stats_workspace(B);
    if (!workspace || workspace_bytes < need || !aligned256(workspace))
        return set_error(ZR_ERR_WORKSPACE, "batch stats workspace needs %zu bytes, 256-aligned", need);
    char* w = static_cast<char*>(workspace);
    int32_t* plen = reinterpret_cast<int32_t*>(w);
    int32_t* rlen = reinterpret_cast<int32_t*>(w + align256((size_t)B * 4));
    int32_t* status = reinterpret_cast<int32_t*>(w + 2 * align256((size_t)B * 4));
    zr_batch_stats* dev = reinterpret_cast<zr_batch_stats*>(w + 2 * align256((size_t)B * 4) + align256(16));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    zr_status st = launch_batch_stats(attention_mask, B, L, L - response_length, plen, rlen, status, dev, s);
    if (st != ZR_OK) return st;
    ZR_CUDA_TRY(cudaMemcpyAsync(out, dev, sizeof(zr_batch_stats), cudaMemcpyDeviceToHost, s));
    ZR_CUDA_TRY(cudaStreamSynchronize(s));
    return ZR_OK;
}

size_t zr_split_attn_workspace(const zr_recon_info* info, int Hq, int /*Hkv*/, int D) {
    if (!info || info->T_cap <= 0 || info->B <= 0 || Hq <= 0) return 0;
    return attn_workspace_layout(*info, Hq, D, nullptr, nullptr);
}

static zr_status attn_common(const zr_recon_info* info, int Hq, int Hkv, int D, zr_dtype dtype,
                             void* workspace, size_t workspace_bytes, AttnWorkspace* ws) {
    zr_status st = check_info(info);
    if (st != ZR_OK) return st;
    if (Hq <= 0 || Hkv <= 0) return set_error(ZR_ERR_INVALID_ARG, "Hq=%d Hkv=%d must be positive", Hq, Hkv);
    if (Hq % Hkv) return set_error(ZR_ERR_UNSUPPORTED, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
    if (dtype != ZR_BF16 && dtype != ZR_F32) return set_error(ZR_ERR_UNSUPPORTED, "dtype %d", (int)dtype);
    if (dtype == ZR_BF16 && D != 64 && D != 128)
        return set_error(ZR_ERR_UNSUPPORTED, "bf16 head_dim %d (the tensor-core kernels take 64 or 128)", D);
    if (dtype == ZR_F32 && D != 32 && D != 64 && D != 96 && D != 128)
        return set_error(ZR_ERR_UNSUPPORTED, "float32 head_dim %d (supported: 32, 64, 96, 128)", D);
    const size_t need = attn_workspace_layout(*info, Hq, D, nullptr, nullptr);
    if (!workspace || workspace_bytes < need || !aligned256(workspace))
        return set_error(ZR_ERR_WORKSPACE, "attention workspace needs %zu bytes, 256-aligned", need);
    attn_workspace_layout(*info, Hq, D, workspace, ws);
    return ZR_OK;
}

zr_status zr_split_attn_fwd(const zr_recon_info* info, const void* q, const void* k, const void* v,
                            void* o, float* lse, int Hq, int Hkv, int D, zr_dtype dtype,
                            float softmax_scale, void* workspace, size_t workspace_bytes,
                            void* stream) {
    ZR_NVTX("zr_split_attn_fwd");
    AttnWorkspace ws;
    zr_status st = attn_common(info, Hq, Hkv, D, dtype, workspace, workspace_bytes, &ws);
    if (st != ZR_OK) return st;
    if (!q || !k || !v || !o || !lse) return set_error(ZR_ERR_INVALID_ARG, "NULL q/k/v/o/lse");
    AttnArgs a = {};
    a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
    a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.dtype = dtype;
    a.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D);
    a.T_cap = info->T_cap;
    // bf16 runs on the tensor cores, float32 on the SIMT kernels (attn_common
    // has rejected every other shape)
    const bool tc = dtype == ZR_BF16;
    if (tc && !tc_fwd_supported(a))
        return set_error(ZR_ERR_UNSUPPORTED, "no tensor-core forward for D=%d Hq=%d Hkv=%d", D, Hq, Hkv);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ZR_CUDA_TRY(cudaMemsetAsync(ws.status, 0, 4 * sizeof(int), s));
    st = launch_attn_plan(*info, ws, s);
    if (st != ZR_OK) return st;
    st = tc ? launch_attn_fwd_tc(*info, ws, a, s) : launch_attn_fwd_simt(*info, ws, a, s);
    if (st != ZR_OK) return st;
    const int64_t e = dtype == ZR_F32 ? 4 : 2;
    st = launch_zero_pad_rows(*info, o, (int64_t)Hq * D * e, s);
    if (st != ZR_OK) return st;
    return launch_zero_pad_rows(*info, lse, (int64_t)Hq * 4, s);
}

zr_status zr_split_attn_bwd(const zr_recon_info* info, const void* q, const void* k, const void* v,
                            const void* o, const float* lse, const void* dout, void* dq, void* dk,
                            void* dv, int Hq, int Hkv, int D, zr_dtype dtype, float softmax_scale,
                            void* workspace, size_t workspace_bytes, void* stream) {
    ZR_NVTX("zr_split_attn_bwd");
    AttnWorkspace ws;
    zr_status st = attn_common(info, Hq, Hkv, D, dtype, workspace, workspace_bytes, &ws);
    if (st != ZR_OK) return st;
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv)
        return set_error(ZR_ERR_INVALID_ARG, "NULL q/k/v/o/lse/dout/dq/dk/dv");
    AttnArgs a = {};
    a.q = q; a.k = k; a.v = v; a.o_in = o; a.lse_in = lse; a.dout = dout;
    a.dq = dq; a.dk = dk; a.dv = dv;
    a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.dtype = dtype;
    a.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D);
    a.T_cap = info->T_cap;
    const bool tc = dtype == ZR_BF16;
    if (tc && !tc_bwd_supported(a))
        return set_error(ZR_ERR_UNSUPPORTED, "no tensor-core backward for D=%d Hq=%d Hkv=%d", D, Hq, Hkv);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ZR_CUDA_TRY(cudaMemsetAsync(ws.status, 0, 4 * sizeof(int), s));
    st = launch_attn_plan(*info, ws, s);
    if (st != ZR_OK) return st;
    if (tc) {
        st = launch_attn_bwd_tc(*info, ws, a, s);  // computes its own head-major Delta
    } else {
        st = launch_attn_delta(*info, ws, a, s);
        if (st == ZR_OK) st = launch_attn_bwd_simt(*info, ws, a, s);
    }
    if (st != ZR_OK) return st;
    const int64_t e = dtype == ZR_F32 ? 4 : 2;
    st = launch_zero_pad_rows(*info, dq, (int64_t)Hq * D * e, s);
    if (st != ZR_OK) return st;
    st = launch_zero_pad_rows(*info, dk, (int64_t)Hkv * D * e, s);
    if (st != ZR_OK) return st;
    return launch_zero_pad_rows(*info, dv, (int64_t)Hkv * D * e, s);
}

zr_status zr_check_status(const zr_recon_info* info, void* attn_workspace, void* stream) {
    ZR_NVTX("zr_check_status");
    zr_status st = check_info(info);
    if (st != ZR_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t hs[4] = {0, 0, 0, 0}, ha[4] = {0, 0, 0, 0};
    ZR_CUDA_TRY(cudaMemcpyAsync(hs, info->status, sizeof(hs), cudaMemcpyDeviceToHost, s));
    AttnWorkspace ws;
    if (attn_workspace) {
        attn_workspace_layout(*info, 1, 0, attn_workspace, &ws);
        ZR_CUDA_TRY(cudaMemcpyAsync(ha, ws.status, sizeof(ha), cudaMemcpyDeviceToHost, s));
    }
    ZR_CUDA_TRY(cudaStreamSynchronize(s));
    ZR_CUDA_TRY(cudaMemsetAsync(info->status, 0, sizeof(hs), s));
    if (attn_workspace) ZR_CUDA_TRY(cudaMemsetAsync(ws.status, 0, sizeof(ha), s));
    if (hs[kStatusMask])
        return set_error(ZR_ERR_INVALID_ARG, "attention_mask layout unsupported: prompts must be "
                         "left padded and responses right padded");
    if (hs[kStatusCapacity]) return set_error(ZR_ERR_CAPACITY, "packed tokens exceed T_cap");
    if (hs[kStatusTimeout])
        return set_error(ZR_ERR_TIMEOUT, "a bounded device wait gave up (code %d)", hs[kStatusTimeout]);
    if (hs[kStatusBounds])
        return set_error(ZR_ERR_INVALID_ARG, "debug bounds check failed at site %d", hs[kStatusBounds]);
    if (ha[kStatusTimeout])
        return set_error(ZR_ERR_TIMEOUT, "a bounded device wait gave up (code %d)", ha[kStatusTimeout]);
    return ZR_OK;
}

}  // extern "C"
