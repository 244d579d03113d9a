// Exact prompt grouping ("How Prompt Deduplication Works", "Finding Prompt
// Groups").
//
// 1. hash_rows: a 64-bit hash of every row's prompt (and prompt mask).  Each
//    position contributes mix(token, position, mask bit) and the contributions
//    are summed modulo 2^64, so chunks of a row hash in parallel and the sum
//    does not depend on the order of the atomic adds.  mix is the SplitMix64
//    finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom number
//    generators", OOPSLA 2014).
// 2. match_rows: row b scans rows a < b in increasing order; at every a with
//    an equal hash it compares the two prompts in full and stops at the first
//    equal one.  Equality is transitive, so the row found is the smallest
//    equal row: rep[b] = min{a : prompt a == prompt b}.  A hash collision only
//    costs an extra comparison; the groups stay exact.
// 3. compact_groups: groups in order of their representative (first
//    occurrence), members ascending, as CSR.
// 4. gather_unique_prompts: unique_prompts[g] = input_ids[rep_g, 0:P].
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "zr_internal.h"

namespace zr {
namespace {

constexpr int kHashChunk = 4096;   // prompt positions per hashing block
constexpr int kCompareChunk = 2048;
constexpr int kMaxGroupRows = 8192;

__device__ __forceinline__ uint64_t splitmix64_finalize(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

__global__ void hash_rows_kernel(const int64_t* __restrict__ ids, const uint8_t* __restrict__ mask,
                                 int L, int P, int weak, unsigned long long* __restrict__ hash) {
    const int b = blockIdx.y;
    const int lo = blockIdx.x * kHashChunk;
    const int hi = min(lo + kHashChunk, P);
    const int64_t* row = ids + (int64_t)b * L;
    const uint8_t* mrow = mask ? mask + (int64_t)b * L : nullptr;
    uint64_t h = 0;
    for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) {
        uint64_t tok = (uint64_t)row[i];
        uint64_t m = mrow ? (mrow[i] != 0 ? 1ull : 2ull) : 1ull;
        h += splitmix64_finalize(tok * 0x9e3779b97f4a7c15ull + (uint64_t)i * 0xd1b54a32d192ed03ull +
                                 m * 0x8cb92ba72f3d8dd7ull);
    }
    // block sum
    for (int o = 16; o > 0; o >>= 1) h += __shfl_xor_sync(0xffffffffu, h, o);
    __shared__ unsigned long long warp_sum[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) warp_sum[warp] = h;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint64_t t = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += warp_sum[w];
        if (weak) t = 0x5bd1e995ull;  // forced collisions: every prompt looks alike
        if (weak) {
            if (blockIdx.x == 0) hash[b] = t;
        } else {
            atomicAdd(&hash[b], (unsigned long long)t);
        }
    }
}

__global__ void match_rows_kernel(const int64_t* __restrict__ ids, const uint8_t* __restrict__ mask,
                                  int B, int L, int P, const unsigned long long* __restrict__ hash,
                                  int32_t* __restrict__ rep) {
    const int b = blockIdx.x;
    const uint64_t hb = hash[b];
    const int64_t* rb = ids + (int64_t)b * L;
    const uint8_t* mb = mask ? mask + (int64_t)b * L : nullptr;
    int result = b;
    for (int a = 0; a < b; ++a) {
        if (hash[a] != hb) continue;  // same value for every thread of the block
        const int64_t* ra = ids + (int64_t)a * L;
        const uint8_t* ma = mask ? mask + (int64_t)a * L : nullptr;
        bool equal = true;
        for (int base = 0; base < P && equal; base += kCompareChunk) {
            const int hi = min(base + kCompareChunk, P);
            int diff = 0;
            for (int i = base + threadIdx.x; i < hi; i += blockDim.x) {
                diff |= (ra[i] != rb[i]);
                if (mask) diff |= ((ma[i] != 0) != (mb[i] != 0));
            }
            equal = !__syncthreads_or(diff);
        }
        if (equal) { result = a; break; }
    }
    if (threadIdx.x == 0) rep[b] = result;
}

// In-place exclusive scan of n ints in shared memory; returns the total.
// Every thread of the block must call it.
__device__ int block_exclusive_scan(int* data, int n) {
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

__global__ void compact_groups_kernel(const int32_t* __restrict__ rep, int B, int32_t* group_ptr,
                                      int32_t* members, int32_t* group_of, int32_t* num_groups) {
    extern __shared__ int smem[];
    int* s_rep = smem;            // [B]
    int* s_gid = smem + B;        // [B]: exclusive scan of "is representative"
    int* s_cnt = smem + 2 * B;    // [B]: members per group, then group_ptr
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        int r = rep[b];
        s_rep[b] = r;
        s_gid[b] = (r == b) ? 1 : 0;
        s_cnt[b] = 0;
    }
    __syncthreads();
    const int G = block_exclusive_scan(s_gid, B);
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        int g = s_gid[s_rep[b]];
        group_of[b] = g;
        atomicAdd(&s_cnt[g], 1);
    }
    __syncthreads();
    block_exclusive_scan(s_cnt, B);  // entries >= G are zero-count groups
    for (int g = threadIdx.x; g <= B; g += blockDim.x)
        group_ptr[g] = (g < G) ? s_cnt[g] : B;
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        const int r = s_rep[b];
        int rank = 0;
        for (int a = r; a < b; ++a) rank += (s_rep[a] == r);  // members precede b
        members[s_cnt[s_gid[r]] + rank] = b;
    }
    if (threadIdx.x == 0) num_groups[0] = G;
}

__global__ void gather_unique_prompts_kernel(const int64_t* __restrict__ ids, int L, int P,
                                             const int32_t* __restrict__ group_ptr,
                                             const int32_t* __restrict__ members,
                                             const int32_t* __restrict__ num_groups,
                                             int64_t* __restrict__ out) {
    const int g = blockIdx.y;
    if (g >= num_groups[0]) return;
    const int r = members[group_ptr[g]];
    const int lo = blockIdx.x * kHashChunk, hi = min(lo + kHashChunk, P);
    for (int i = lo + threadIdx.x; i < hi; i += blockDim.x)
        out[(int64_t)g * P + i] = ids[(int64_t)r * L + i];
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

size_t group_workspace_bytes(int B, int /*L*/) {
    return align256((size_t)B * 8) + align256((size_t)B * 4);
}

zr_status launch_find_groups(const int64_t* ids, const uint8_t* mask, int B, int L, int P,
                             const zr_groups& out, int64_t* unique_prompts, void* ws,
                             cudaStream_t s) {
    if (B > kMaxGroupRows) return set_error(ZR_ERR_UNSUPPORTED, "B=%d exceeds %d rows", B, kMaxGroupRows);
    unsigned long long* hash = reinterpret_cast<unsigned long long*>(ws);
    int32_t* rep = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(ws) + align256((size_t)B * 8));
    ZR_CUDA_TRY(cudaMemsetAsync(hash, 0, (size_t)B * 8, s));
    const int nchunk = P > 0 ? (P + kHashChunk - 1) / kHashChunk : 1;
    hash_rows_kernel<<<dim3(nchunk, B), 256, 0, s>>>(ids, mask, L, P, options().weak_hash, hash);
    ZR_LAUNCH_CHECK("hash_rows_kernel");
    match_rows_kernel<<<B, 256, 0, s>>>(ids, mask, B, L, P, hash, rep);
    ZR_LAUNCH_CHECK("match_rows_kernel");
    const size_t smem = (size_t)3 * B * sizeof(int);
    // the attribute belongs to the current device; setting it on every call is
    // a cheap host call and needs no per-device or cross-thread bookkeeping
    ZR_CUDA_TRY(cudaFuncSetAttribute(compact_groups_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     3 * kMaxGroupRows * (int)sizeof(int)));
    compact_groups_kernel<<<1, 1024, smem, s>>>(rep, B, out.group_ptr, out.members, out.group_of,
                                                out.num_groups);
    ZR_LAUNCH_CHECK("compact_groups_kernel");
    if (unique_prompts && P > 0) {
        gather_unique_prompts_kernel<<<dim3(nchunk, B), 256, 0, s>>>(
            ids, L, P, out.group_ptr, out.members, out.num_groups, unique_prompts);
        ZR_LAUNCH_CHECK("gather_unique_prompts_kernel");
    }
    return ZR_OK;
}

}  // namespace zr

// ---------------------------------------------------------------------------
// Allocation-free grouping.  Some callers cannot hand this library a
// workspace: for example a plug-in that is given only borrowed device
// buffers by a host framework which owns every allocation, or code that runs
// under a hard device-memory budget where no allocator call may be made.
// For them, zr_find_prompt_groups_noalloc keeps its scratch (the row hashes
// and representatives) in a fixed array in device memory that is part of the
// library image: every GPU that loads the library holds these 48 KiB until
// the process exits.
namespace zr {
namespace {

constexpr int kNoAllocMaxRows = 4096;
constexpr size_t kNoAllocScratchBytes = ((size_t)kNoAllocMaxRows * 8 + 255) / 256 * 256 +
                                        ((size_t)kNoAllocMaxRows * 4 + 255) / 256 * 256;

static __device__ __align__(256) unsigned char g_group_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 256;

// The cached device address of g_group_scratch, per device, together with the
// unique ID of the CUDA context it was looked up in.  A device reset
// (cudaDeviceReset) destroys that context and the array with it; the next
// call sees a new context ID and looks the address up again.
struct ScratchCache {
    unsigned long long ctx_id = 0;
    void* addr = nullptr;
};
ScratchCache g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique ID of the calling thread's current context (0 if it cannot be read).
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_group_scratch on the current device.  The host-side
// name is only a stand-in, so the address is looked up with the device current
// (cudaGetSymbolAddress), once per device and context, and cached.  When the
// context ID cannot be read the look-up runs on every call.
zr_status scratch_address(void** out) {
    int dev = 0;
    ZR_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return set_error(ZR_ERR_UNSUPPORTED, "device index %d", dev);
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    ScratchCache& c = g_scratch[dev];
    if (!c.addr || id == 0 || c.ctx_id != id) {
        void* p = nullptr;
        ZR_CUDA_TRY(cudaGetSymbolAddress(&p, g_group_scratch));
        c.addr = p;
        c.ctx_id = id;
    }
    *out = c.addr;
    return ZR_OK;
}

}  // namespace
}  // namespace zr

extern "C" zr_status zr_find_prompt_groups_noalloc(const int64_t* input_ids, const uint8_t* attention_mask,
                                                   int B, int L, int response_length, const zr_groups* out,
                                                   int64_t* unique_prompts, int32_t* num_groups_host,
                                                   void* stream) {
    using namespace zr;
    ZR_NVTX("zr_find_prompt_groups_noalloc");
    if (!input_ids || !out || !out->group_ptr || !out->members || !out->group_of || !out->num_groups)
        return set_error(ZR_ERR_INVALID_ARG, "NULL input_ids or group output");
    if (B <= 0 || L <= 0) return set_error(ZR_ERR_INVALID_ARG, "B and L must be positive (B=%d L=%d)", B, L);
    if (response_length < 0 || response_length > L)
        return set_error(ZR_ERR_INVALID_ARG, "response_length %d outside [0, L=%d]", response_length, L);
    if (B > kNoAllocMaxRows)
        return set_error(ZR_ERR_UNSUPPORTED,
                         "zr_find_prompt_groups_noalloc handles at most %d rows (B=%d); use "
                         "zr_find_prompt_groups with a workspace",
                         kNoAllocMaxRows, B);
    void* scratch = nullptr;
    zr_status st = scratch_address(&scratch);
    if (st != ZR_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // launch_find_groups clears the hash accumulators it needs at zero
    st = launch_find_groups(input_ids, attention_mask, B, L, L - response_length, *out, unique_prompts,
                            scratch, s);
    if (st != ZR_OK) return st;
    if (num_groups_host) {
        ZR_CUDA_TRY(cudaMemcpyAsync(num_groups_host, out->num_groups, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
        ZR_CUDA_TRY(cudaStreamSynchronize(s));
    }
    return ZR_OK;
}

namespace zr {
namespace {
// Every row its own group: group_ptr[i] = i, members[i] = group_of[i] = i.
__global__ void identity_groups_kernel(int B, int32_t* __restrict__ group_ptr, int32_t* __restrict__ members,
                                       int32_t* __restrict__ group_of, int32_t* __restrict__ num_groups) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i <= B) group_ptr[i] = i;
    if (i < B) {
        members[i] = i;
        group_of[i] = i;
    }
    if (i == 0) num_groups[0] = B;
}
}  // namespace
}  // namespace zr

extern "C" zr_status zr_identity_groups(int B, const zr_groups* out, void* stream) {
    using namespace zr;
    ZR_NVTX("zr_identity_groups");
    if (!out || !out->group_ptr || !out->members || !out->group_of || !out->num_groups)
        return set_error(ZR_ERR_INVALID_ARG, "NULL group output");
    if (B <= 0) return set_error(ZR_ERR_INVALID_ARG, "B must be positive (B=%d)", B);
    if (B > 8192) return set_error(ZR_ERR_UNSUPPORTED, "B=%d exceeds 8192 rows", B);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    identity_groups_kernel<<<(B + 256) / 256, 256, 0, s>>>(B, out->group_ptr, out->members, out->group_of,
                                                            out->num_groups);
    ZR_LAUNCH_CHECK("identity_groups_kernel");
    return ZR_OK;
}
