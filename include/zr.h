/*
 * zr.h -- C ABI of the prompt-deduplication hot path (libzr).
 *
 * The calls follow the problem statement of "How Prompt Deduplication Works"
 * (trybrowzer.com/help/snowflake-research/how-prompt-deduplication-works):
 * input_ids [B, L] plus response_length go in; prompt groups, the unique
 * prompts, one packed [1, T] sequence and reconstruction info come out; split
 * attention runs forward and backward on the packed sequence; reconstruction
 * scatters packed rows back to [B, L, hidden].
 *
 * Conventions shared by every call
 *  - Every pointer argument is DEVICE memory owned by the caller unless it is
 *    marked "host".  The library allocates no memory and keeps no state
 *    between calls apart from the options set with zr_set_option.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *    asynchronous on that stream; the only host synchronisations are the
 *    optional host read-backs named in a call (num_groups_host, T_host) and
 *    zr_check_status.
 *  - Arguments are validated on the host before any launch: a call that
 *    returns ZR_ERR_INVALID_ARG, ZR_ERR_UNSUPPORTED or ZR_ERR_WORKSPACE has
 *    launched nothing.  The one status found after launching is the
 *    ZR_ERR_CAPACITY of zr_pack_dedup with a host read-back (its plan kernel
 *    has run; nothing was gathered).  Kernel launch errors are ZR_ERR_CUDA.
 *    Conditions that only the device can see (an unsupported mask layout, a
 *    packed capacity that is too small, a bounded wait that ran out) are
 *    written to the device status words of the reconstruction info and
 *    reported by zr_check_status.
 *  - No C++ exception crosses this interface.
 *  - The row tensors are token-major and contiguous:
 *      q, o, dq, dout : [T_cap, Hq, D]      k, v, dk, dv : [T_cap, Hkv, D]
 *      lse            : [T_cap, Hq] float32 (natural-log log-sum-exp)
 *    Only the first T rows (T = packed token count) are read or written.
 */
#ifndef ZR_H_
#define ZR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ZR_OK = 0,
    ZR_ERR_INVALID_ARG = 1,     /* bad pointer, size or layout */
    ZR_ERR_UNSUPPORTED = 2,     /* valid but not implemented (dtype, head_dim, sizes) */
    ZR_ERR_CAPACITY = 3,        /* packed tokens exceed the caller's capacity */
    ZR_ERR_WORKSPACE = 4,       /* workspace missing or too small */
    ZR_ERR_CUDA = 5,            /* a CUDA runtime call failed */
    ZR_ERR_TIMEOUT = 6,         /* a bounded device wait gave up (kernel exited cleanly) */
    ZR_ERR_NOT_IMPLEMENTED = 7
} zr_status;

typedef enum { ZR_BF16 = 0, ZR_F32 = 1 } zr_dtype;

/* Message for the last non-OK status returned on the calling host thread.
 * Valid until the next zr_* call on that thread; never NULL. */
const char* zr_last_error(void);

/* ABI version of this header (major * 100 + minor). */
int zr_version(void);

/* 1 in the debug build (libzr_debug.so, compiled with ZR_DEBUG_BOUNDS), else
 * 0.  The debug build checks every global row index that a kernel derives
 * from the device-built plans (pack and reconstruction segments, attention
 * query blocks and key tiles) before the access; a failed check skips the
 * access and records its site in the reconstruction info's status words,
 * which zr_check_status reports as ZR_ERR_INVALID_ARG ("debug bounds check
 * failed at site N").  Same ABI and results as libzr.so otherwise. */
int zr_debug_bounds(void);

/* Number of kernels this library has launched in this process (all devices),
 * for launch accounting in benchmarks. */
int64_t zr_kernel_launches(void);

/* Test and tuning knobs (process-wide, not thread-safe; set before use):
 *  "weak_hash"   1 = every prompt hashes to the same value (forces the exact
 *                row comparison to resolve all groups; results are unchanged)
 *  "wait_limit"  bounded-wait limit of the tensor-core kernels in SM clock
 *                cycles (0 = default, 4e9 cycles: about two seconds)
 *  "test_withhold_arrival"  test option: bit 0 makes the forward skip the
 *                Q load of its first work unit, bit 1 makes the backward skip
 *                the K/V load of its first work unit (in whichever CTA takes
 *                that unit).  The wait on that load runs out
 *                after "wait_limit" cycles, the CTA leaves cleanly and
 *                zr_check_status reports ZR_ERR_TIMEOUT; the outputs of that
 *                call are incomplete.  0 = off (the only production value)
 *  "kernel_timing" 1 = record a CUDA event pair on the launch stream around
 *                every launch of the kernels named under zr_kernel_time
 *                (a few microseconds of host work per launch; 0 = off)
 * Returns ZR_ERR_INVALID_ARG for an unknown name. */
zr_status zr_set_option(const char* name, int64_t value);

/* Per-kernel device time, for roofline reporting.  While the "kernel_timing"
 * option is on, each launch of the kernels below is bracketed by two CUDA
 * events recorded on the stream it is launched on.  zr_kernel_time waits for
 * the recorded pairs filed under `name` and returns their summed elapsed time
 * in milliseconds and their count.  Names: "attn_fwd", "attn_bwd_prep",
 * "attn_bwd", "attn_dq_convert" (tensor-core attention), "pack_gather",
 * "reconstruct", "reconstruct_backward", "pack_backward",
 * "reconstruct_pack_backward" (row copies).  An unknown name yields 0
 * launches.
 * At most 16384 pairs are kept; pairs past that are dropped and the call
 * returns ZR_ERR_CAPACITY (with the sums of the kept pairs written).
 * zr_kernel_time_reset waits for and forgets every recorded pair.  Both are
 * host calls that block; neither launches a kernel.  This library feature is
 * instrumentation with no counterpart on the pages. */
zr_status zr_kernel_time(const char* name, double* total_ms, int64_t* launches);
zr_status zr_kernel_time_reset(void);

/* -------------------------------------------------------------------------
 * Finding prompt groups ("Finding Prompt Groups"; "Phase 1: Prompt Detection
 * & Deduplication").
 *
 * The prompt of row b is input_ids[b, 0:P] with P = L - response_length; with
 * an attention mask the key also includes mask[b, 0:P].  Rows with equal keys
 * form a group.  Groups are ordered by their smallest member and members are
 * ascending (the page's example [[0,1],[2,3]]).  Grouping is exact: a 64-bit
 * hash selects candidates and a full row comparison decides.
 *
 *  input_ids       [B, L] int64 (device)
 *  attention_mask  [B, L] uint8, 1 = token, 0 = pad; NULL = all tokens
 *  out->group_ptr  [B+1] int32: group g's members are
 *                  members[group_ptr[g] .. group_ptr[g+1])
 *  out->members    [B]   int32
 *  out->group_of   [B]   int32: group of row b
 *  out->num_groups [1]   int32: G
 *  unique_prompts  [B, P] int64 capacity, first G rows written; may be NULL
 *  num_groups_host host int32*, may be NULL; if set the call synchronises
 *                  the stream and stores G there
 *  workspace       zr_find_prompt_groups_workspace(B, L) bytes, 256-aligned
 * Limits: 1 <= B <= 8192, 0 <= response_length <= L.
 */
typedef struct {
    int32_t* group_ptr;
    int32_t* members;
    int32_t* group_of;
    int32_t* num_groups;
} zr_groups;

size_t zr_find_prompt_groups_workspace(int B, int L);
zr_status zr_find_prompt_groups(const int64_t* input_ids, const uint8_t* attention_mask,
                                int B, int L, int response_length,
                                const zr_groups* out, int64_t* unique_prompts,
                                int32_t* num_groups_host,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Allocation-free variant of zr_find_prompt_groups (the pages have no
 * counterpart; this is an interface convenience).  It is for callers that
 * cannot hand the library a workspace at all -- for example a plug-in given
 * only borrowed device buffers by a host framework that owns every
 * allocation, or code running under a hard device-memory budget where no
 * allocator may be called.  Its scratch is a fixed 48 KiB array in device
 * memory that belongs to the library image: every GPU that loads libzr holds
 * it until the process exits.  The call itself allocates nothing.
 *
 * Same arguments, results and errors as zr_find_prompt_groups, without the
 * workspace.  Limit: B <= 4096 rows (larger B returns ZR_ERR_UNSUPPORTED
 * before any launch).  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture.  The address is cached per device
 * together with the ID of the CUDA context it belongs to: after a
 * cudaDeviceReset the next call on that device sees a new context and repeats
 * the look-up, so that call, too, belongs before any stream capture.  Every call on a device shares the
 * one array, which keeps the previous call's contents (the call clears what
 * must start at zero): calls that can overlap on the GPU -- on different
 * streams, or from different host threads -- race and must be serialised by
 * the caller. */
zr_status zr_find_prompt_groups_noalloc(const int64_t* input_ids, const uint8_t* attention_mask,
                                        int B, int L, int response_length,
                                        const zr_groups* out, int64_t* unique_prompts,
                                        int32_t* num_groups_host, void* stream);

/* Every row its own group (group_ptr[i] = i, members[i] = group_of[i] = i,
 * num_groups = B), without looking at the tokens.  With this grouping,
 * zr_pack_dedup keeps every row's prompt (use_unpad = 0: the packed layout is
 * the [B, L] rows back to back) and zr_split_attn_* compute ordinary causal
 * attention over each full sequence: the "standard QKV" strategy of "Split
 * Attention Optimization" (reconstruct Q, K, V, then plain attention), and
 * the no-deduplication baseline.  B <= 8192.  Async on `stream`. */
zr_status zr_identity_groups(int B, const zr_groups* out, void* stream);

/* -------------------------------------------------------------------------
 * Reconstruction info ("Creating Deduplicated Batch": reconstruction_info;
 * "Working with Packed/Unpacked Sequences": padding boundaries).  The layout is
 * this library's.  All arrays live in ONE caller buffer of
 * zr_recon_info_bytes(B) bytes that zr_recon_info_bind carves up; the host
 * fields describe the batch.  zr_pack_dedup fills the arrays.
 *
 *  prompt_off[g]  packed row where group g's prompt slot starts
 *  prompt_slot[g] rows in that slot: P (padded) or the valid prompt tokens
 *                 (use_unpad)
 *  prompt_len[g]  valid prompt tokens of the group
 *  resp_off[b]    packed row where sample b's response slot starts
 *  resp_slot[b]   rows in that slot: R (padded) or the valid tokens (use_unpad)
 *  resp_len[b]    valid response tokens of sample b
 *  group_ptr, members, group_of, num_groups: copies of the grouping
 *  total_tokens   [1] T
 *  status         [4] device status words (see zr_check_status)
 *
 * Mask layout: within a row the prompt must be left padded (zeros then ones)
 * and the response right padded (ones then zeros).  Other layouts set
 * status[0] = ZR_ERR_INVALID_ARG and T = 0, after which every later call on
 * that info writes nothing.
 */
typedef struct {
    int32_t* prompt_off;
    int32_t* prompt_slot;
    int32_t* prompt_len;
    int32_t* resp_off;
    int32_t* resp_slot;
    int32_t* resp_len;
    int32_t* group_ptr;
    int32_t* members;
    int32_t* group_of;
    int32_t* num_groups;
    int32_t* total_tokens;
    int32_t* status;
    int64_t* pack_segs;     /* internal: [2B][3] row-copy segments of the pack */
    int64_t* recon_segs;    /* internal: [4B][3] row-copy segments of reconstruction */
    int64_t* pad_segs;      /* internal: [2B][3] pad-row segments (zero fill) */
    int32_t* row_prompt_len;/* internal: [B] valid prompt tokens of every row */
    int64_t* pack_order;    /* internal: [2B][3] the pack segments sorted by packed row */
    int B, L, P, use_unpad;
    int64_t T_cap;          /* rows of every packed buffer */
} zr_recon_info;

size_t zr_recon_info_bytes(int B);
/* Point the arrays of *info into `buffer` (device, zr_recon_info_bytes(B)
 * bytes, 256-aligned) and set the host fields.  No launch, no sync. */
zr_status zr_recon_info_bind(zr_recon_info* info, void* buffer, int B, int L,
                             int response_length, int use_unpad, int64_t T_cap);

/* -------------------------------------------------------------------------
 * Creating the deduplicated batch ("Creating Deduplicated Batch").
 *
 * Packs every row into one sequence laid out as
 * [Prompt_1][Response_1_1][Response_1_2]...[Prompt_2][Response_2_1]...
 * Each group's prompt is taken once from its first member; each member's
 * response follows in member order.  use_unpad = 0 keeps all P prompt and R
 * response positions (pads included); use_unpad = 1 keeps only mask = 1
 * positions.  Position ids are copied from the source rows.
 *
 *  input_ids, position_ids [B, L] int64 (position_ids NULL: not packed)
 *  attention_mask          [B, L] uint8 or NULL
 *  groups                  the output of zr_find_prompt_groups
 *  dedup_input_ids         [T_cap] int64; dedup_position_ids [T_cap] int64 or NULL
 *  dedup_mask              [T_cap] uint8 or NULL: the packed attention mask
 *  info                    bound with zr_recon_info_bind (B, L, response
 *                          length, use_unpad, T_cap); its arrays are filled
 *  T_host                  host int64*, may be NULL; if set the call
 *                          synchronises and stores T, and returns
 *                          ZR_ERR_CAPACITY when T > T_cap (nothing gathered)
 * Without T_host a too-small T_cap is reported through status[1] and only the
 * rows that fit are written.  T_cap = B * L always suffices.
 */
zr_status zr_pack_dedup(const int64_t* input_ids, const int64_t* position_ids,
                        const uint8_t* attention_mask, const zr_groups* groups,
                        int64_t* dedup_input_ids, int64_t* dedup_position_ids,
                        uint8_t* dedup_mask, zr_recon_info* info, int64_t* T_host,
                        void* stream);

/* Apply the same gather to any [B, L, row_bytes] row tensor (hidden states):
 * src [B, L] rows of row_bytes bytes -> dst [T_cap] rows. */
zr_status zr_pack_rows(const zr_recon_info* info, const void* src, int64_t row_bytes,
                       void* dst, void* stream);

/* -------------------------------------------------------------------------
 * Reconstructing the original batch ("Reconstructing Original Batch"): for
 * each sample copy its group's prompt, then its own response rows, from the
 * packed [T, row_bytes] tensor into out [B, L, row_bytes].  Positions that no
 * packed row maps to (pads dropped by use_unpad) are zero-filled.
 */
zr_status zr_reconstruct(const zr_recon_info* info, const void* packed, int64_t row_bytes,
                         void* out, void* stream);

/* The adjoint of zr_reconstruct, for the backward pass through the
 * reconstruction ("Correctness & Gradients": a shared prompt's gradient
 * collects the contributions of all responses of its group).  Packed row t
 * receives the sum, over every output position zr_reconstruct copies it to,
 * of grad_out there: a group's prompt rows sum the gradients of all members'
 * prompt copies (fp32 accumulation in group-member order, rounded once to the
 * element type), a response row takes its own sample's gradient.  Positions
 * that zr_reconstruct zero-fills contribute nothing.
 *  grad_out     [B, L, W] elements of `dtype` (ZR_BF16 or ZR_F32), device
 *  grad_packed  [T_cap, W] elements of `dtype`, device; rows [0, T) written,
 *               rows [T, T_cap) untouched
 * Returns ZR_ERR_UNSUPPORTED for other element types.  Async on `stream`. */
zr_status zr_reconstruct_backward(const zr_recon_info* info, const void* grad_out, int64_t W, int dtype,
                                  void* grad_packed, void* stream);

/* The adjoint of zr_pack_rows / the pack of zr_pack_dedup ("Correctness &
 * Gradients": gradients flow back through the deduplication step as well as
 * the reconstruction).  Source position (b, p) receives the gradient of the
 * packed row that was read from it; each position is read at most once, so
 * this is a copy (any element type, rows of row_bytes bytes).  Positions the
 * pack never read -- the prompt rows of every group member other than its
 * representative (the first member), and the pads that use_unpad dropped --
 * are zero-filled.
 *  grad_packed  [T_cap, row_bytes] device; rows [0, T) read
 *  grad_src     [B, L, row_bytes] device; every position written
 * Async on `stream`. */
zr_status zr_pack_rows_backward(const zr_recon_info* info, const void* grad_packed, int64_t row_bytes,
                                void* grad_src, void* stream);

/* The gradient of zr_reconstruct(zr_pack_rows(x)) with respect to x, in one
 * pass without the packed intermediate: the composition of
 * zr_reconstruct_backward and zr_pack_rows_backward, for a tensor that enters
 * the deduplicated section packed and leaves it reconstructed unchanged (a
 * skip connection around it).  The representative's prompt positions that
 * the pack read receive the fp32 sum, over the group's members in group
 * order, of grad_out there, rounded once to the element type; every row's
 * packed response positions pass their own gradient through; all other
 * positions are zero.  Bitwise equal to the two calls in sequence.
 *  grad_out  [B, L, W] elements of `dtype` (ZR_BF16 or ZR_F32), device
 *  grad_in   [B, L, W] of the same type, device; must not alias grad_out
 * Async on `stream`. */
zr_status zr_reconstruct_pack_backward(const zr_recon_info* info, const void* grad_out, int64_t W,
                                       int dtype, void* grad_in, void* stream);

/* -------------------------------------------------------------------------
 * Batch statistics of a normal (not deduplicated) batch ("Debugging &
 * Analysis", "Batch Statistics"): prompt length, response count with
 * min / mean / max response length, and non-pad tokens with their share of
 * the B * L positions.  Row b's prompt is its first L - response_length
 * positions, its response the rest; a row counts as a response when it holds
 * at least one valid response token, and the response min / mean / max run
 * over those rows (0 when there are none).  This library's reading of the
 * page's one-line summary.
 *  attention_mask  [B, L] uint8 on the device, or NULL (every position valid)
 *  out             host struct, written after one stream synchronisation
 *  workspace       device, zr_batch_stats_workspace(B) bytes, 256-aligned
 */
typedef struct {
    int64_t rows, responses, non_pad_tokens, total_positions;
    int64_t prompt_len_min, prompt_len_max, resp_len_min, resp_len_max;
    double prompt_len_mean, resp_len_mean, non_pad_fraction;
} zr_batch_stats;

size_t zr_batch_stats_workspace(int B);
zr_status zr_batch_stats_compute(const uint8_t* attention_mask, int B, int L, int response_length,
                                 zr_batch_stats* out, void* workspace, size_t workspace_bytes,
                                 void* stream);

/* -------------------------------------------------------------------------
 * Split attention ("Split Attention Optimization": prompt-to-prompt computed
 * once per unique prompt, response-to-full for each response), forward and
 * backward, with grouped-query attention (query head h reads key/value head
 * h / (Hq / Hkv)).
 *
 * A prompt row attends its group's valid prompt rows up to itself.  A
 * response row attends all of its group's valid prompt rows and its own valid
 * response rows up to itself.  Pad rows (mask 0) are never attended; their
 * outputs, LSE and gradients are written as zero.
 *
 *  dtype         ZR_BF16: bf16 in/out with fp32 accumulation, on the
 *                tensor-core kernels (every GQA ratio, MHA included);
 *                ZR_F32: float32 in/out, on the SIMT (CUDA-core) kernels
 *  D             head dimension: 64 or 128 for ZR_BF16; 32, 64, 96 or 128
 *                for ZR_F32 (other values: ZR_ERR_UNSUPPORTED)
 *  softmax_scale <= 0 selects 1/sqrt(D)
 *  workspace     zr_split_attn_workspace(info, Hq, Hkv, D) bytes, 256-aligned;
 *                it includes the backward's fp32 dQ accumulator
 *                (T_cap rounded up to 4, times Hq * D * 4 bytes)
 * The backward takes o and lse from the forward and recomputes the attention
 * probabilities from lse.  Its dQ sums fp32 partials from different key
 * tiles in arrival order, so the last bits of dq can differ between runs;
 * o, lse, dk and dv are bitwise reproducible.
 */
size_t zr_split_attn_workspace(const zr_recon_info* info, int Hq, int Hkv, int D);

zr_status zr_split_attn_fwd(const zr_recon_info* info, const void* q, const void* k,
                            const void* v, void* o, float* lse, int Hq, int Hkv, int D,
                            zr_dtype dtype, float softmax_scale,
                            void* workspace, size_t workspace_bytes, void* stream);

zr_status zr_split_attn_bwd(const zr_recon_info* info, const void* q, const void* k,
                            const void* v, const void* o, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv,
                            int Hq, int Hkv, int D, zr_dtype dtype, float softmax_scale,
                            void* workspace, size_t workspace_bytes, void* stream);

/* -------------------------------------------------------------------------
 * Synchronise `stream` and report the device status words of `info` and of
 * the attention workspace (may be NULL): ZR_ERR_INVALID_ARG (mask layout),
 * ZR_ERR_CAPACITY (T > T_cap) or ZR_ERR_TIMEOUT (a bounded wait gave up),
 * else ZR_OK.  Clears the words it reports.
 */
zr_status zr_check_status(const zr_recon_info* info, void* attn_workspace, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ZR_H_ */
