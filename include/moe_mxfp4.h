/*
 * moe_mxfp4.h — C ABI of the GB300 (sm_103a) MXFP4 mixture-of-experts layer.
 *
 * The layer (one call of each, in order, on one stream):
 *   moe_route          top-k expert routing over fp32 router logits
 *   moe_permute        per-expert histogram, prefix offsets, block-padded
 *                      offsets and the stable token permutation
 *   moe_mxfp4_forward  gather -> grouped W13 GEMM with SiLU(gate)*up ->
 *                      grouped W2 GEMM -> routing-weighted combine
 * plus the one-time weight reorder moe_mxfp4_prepack.
 *
 * The method follows "DeepSeek V4 Flash 单卡 MI300X: 10 个 overlay 起家..."
 * (txtmix.com): §一 (top-6 of 256 experts; routing, then the expert GEMMs),
 * §三 (MXFP4 expert weights with a shared E8M0 scale; the routing bitmatrix
 * whose padding lanes are masked by the logical block size; SiLU fused with a
 * gate/up pair), §九 (the optional SwiGLU clamp). Element formats are the OCP
 * Microscaling (MX) v1.0 E2M1 and E8M0 encodings.
 *
 * Conventions for every entry point:
 *   - Pointers named d_* are DEVICE pointers (cudaMalloc'd or equivalent) on
 *     the current device; the caller allocates and owns all of them. The
 *     library never allocates, frees or keeps device memory between calls.
 *     Every device pointer must be 16-byte aligned; the forward's workspace
 *     256-byte aligned (as cudaMalloc returns it).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). All work is enqueued on that stream only; no call
 *     synchronises the device or copies between host and device (except
 *     moe_read_device_error), so route/permute/forward can be captured in a
 *     CUDA graph. Kernels after the first of a call (and the first kernel of
 *     moe_mxfp4_forward / moe_permute) are launched with programmatic stream
 *     serialization: each may start while the kernel before it on the stream
 *     finishes, and reads or writes nothing that earlier work touches before
 *     that earlier work has completed (griddepcontrol.wait).
 *   - Argument errors are detected on the host before any launch and return
 *     MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_MISALIGNED /
 *     MOE_ERR_WORKSPACE. A failed launch returns MOE_ERR_CUDA. Faults found on
 *     the device (an expert id outside [0,E), a pipeline wait that ran out of
 *     time) never trap: the kernel records a moe_status_t code in a device
 *     error word and skips the faulty access; moe_read_device_error reads it.
 *   - T == 0 is a valid no-op. Logits must be finite and scale bytes must not
 *     be 0xFF (E8M0 NaN); outside these preconditions results are unspecified
 *     but no out-of-bounds access happens.
 */
#ifndef MOE_MXFP4_H
#define MOE_MXFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 4

/* Size of the static scratch array behind moe_mxfp4_forward_noalloc. */
#define MOE_NOALLOC_SCRATCH_BYTES (32u << 20)

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* bad size, null pointer, k > E, ...          */
    MOE_ERR_UNSUPPORTED = 2,   /* valid but outside the shapes this build runs */
    MOE_ERR_MISALIGNED = 3,    /* a pointer is not 16-byte aligned             */
    MOE_ERR_WORKSPACE = 4,     /* workspace or packed buffer too small         */
    MOE_ERR_CUDA = 5,          /* a CUDA runtime/driver call or launch failed  */
    MOE_ERR_DEVICE = 6,        /* device-detected bad input (expert id range)  */
    MOE_ERR_TIMEOUT = 7        /* a bounded device-side wait gave up           */
} moe_status_t;

/* Shapes of one MoE layer.
 *   T tokens, H hidden width, I expert intermediate width, E experts, k
 *   experts per token, block_m the row alignment of each expert segment in
 *   the permutation (16, 32, 64 or 128).
 *   swiglu_limit > 0 enables the clamp gate = min(gate, L),
 *   up = clamp(up, -L, L) before SiLU(gate) * up; <= 0 disables it.
 *   out_dtype: MOE_OUT_F32 (y fp32, the default) or MOE_OUT_BF16 (y as bf16
 *   bits: the fp32 sum of the slot-ordered combine rounded to nearest even).
 *   flags: 0 or MOE_FLAG_FAST_COMBINE.
 * Supported: 1 <= k <= min(E, 32), E <= 1024, H and I multiples of 128. */

/*
 * MOE_FLAG_FAST_COMBINE: permits the W2 GEMM to add w[t,j] * o_j straight
 * into y with fp32 reduction atomics (red.global.add) instead of writing
 * per-pair rows that a separate kernel sums in slot order; y is then zeroed by
 * the forward first. This saves the per-pair rows' round trip and one launch.
 * The library takes it where it is faster: batches of up to 16 rows per
 * expert on average (T*k/E <= 16, the decode shapes); larger batches keep the
 * slot-ordered combine with or without the flag. With the atomic combine the
 * sum order depends on the order the GPU retires the adds: results match the
 * default path up to fp32 rounding (a few ulp of y) and are not
 * bit-reproducible from run to run. The default (flags 0) is always the
 * deterministic slot-ordered combine, and so is MOE_OUT_BF16 output.
 */
#define MOE_FLAG_FAST_COMBINE 1u

typedef enum { MOE_OUT_F32 = 0, MOE_OUT_BF16 = 1 } moe_out_dtype_t;

typedef struct moe_layer_desc {
    int T, H, I, E, k, block_m;
    float swiglu_limit;
    int out_dtype;        /* moe_out_dtype_t */
    unsigned flags;
} moe_layer_desc;

/* ABI version of the loaded library (MOE_ABI_VERSION at build time). */
int moe_abi_version(void);

/* Static description of a status code. */
const char *moe_status_string(moe_status_t status);

/*
 * Routing (txtmix.com §一: every token picks k of E experts from its router
 * scores; §三: the routing bitmatrix).
 *   d_logits    fp32 [T, E] row-major, finite.
 *   d_topk_ids  int32 [T, k] out: the k largest logits of each row in
 *               descending order; equal logits go to the lower expert index
 *               and -0.0 equals +0.0. Bit-exact with the oracle.
 *   d_topk_w    fp32 [T, k] out: softmax over the row restricted to the chosen
 *               k and renormalised (sums to 1).
 *   d_bitmatrix uint32 [T, ceil(E/32)] out, may be NULL: bit (e % 32) of word
 *               e / 32 set iff expert e was chosen; bits >= E are 0.
 * Supported: E <= 1024, 1 <= k <= min(E, 32).
 */
moe_status_t moe_route(const float *d_logits, int T, int E, int k,
                       int32_t *d_topk_ids, float *d_topk_w, uint32_t *d_bitmatrix,
                       void *stream);

/* Rows of the padded permutation: T*k + min(E, T*k) * (block_m - 1). */
int64_t moe_permute_rows_capacity(int T, int E, int k, int block_m);

/*
 * Device workspace bytes moe_permute needs for these sizes: always 0. The
 * permutation keeps its histograms and scans in shared memory, and above 2,048
 * pairs its per-chunk counts in d_pair_to_row until it overwrites them, so the
 * caller passes no workspace; the function exists so that callers written
 * against a workspace-taking permutation can size one without special cases.
 */
size_t moe_permute_workspace_size(int T, int E, int k, int block_m);

/*
 * Permutation (txtmix.com §三: the per-expert histogram whose padding lanes
 * are masked by the logical block size, so lanes past the T*k real (token,
 * slot) pairs never count). Pair p = t*k + j is token t's j-th choice.
 *   d_topk_ids       int32 [T, k] in (from moe_route).
 *   d_counts         int32 [E] out: pairs routed to each expert.
 *   d_offsets        int32 [E+1] out: exclusive prefix sum of counts.
 *   d_padded_offsets int32 [E+1] out: exclusive prefix sum of counts rounded
 *                    up to block_m.
 *   d_row_to_pair    int32 [moe_permute_rows_capacity(...)] out: the rows of
 *                    expert e are padded[e] .. padded[e]+counts[e]-1 holding
 *                    its pairs in ascending pair (= token) order; all other
 *                    rows, padding and tail, hold -1.
 *   d_pair_to_row    int32 [T*k] out: inverse map.
 *   d_error          int32 [1] device error word, may be NULL: set to
 *                    MOE_ERR_DEVICE if an id is outside [0, E) (that pair is
 *                    skipped and its pair_to_row entry is -1).
 * All integer outputs are bit-exact with the oracle. Runs as one thread block
 * up to 2,048 pairs. Above, three launches on chunks of consecutive pairs
 * (chunk histograms, a per-expert scan over the chunks, the scatter); between
 * the first and the last of them d_pair_to_row holds the chunks' counts, so
 * its contents are defined only once the call's work has completed.
 */
moe_status_t moe_permute(const int32_t *d_topk_ids, int T, int E, int k, int block_m,
                         int32_t *d_counts, int32_t *d_offsets, int32_t *d_padded_offsets,
                         int32_t *d_row_to_pair, int32_t *d_pair_to_row, int32_t *d_error,
                         void *stream);

/*
 * moe_route followed by moe_permute on the ids it writes, in one launch (one
 * thread block) for T <= 128 and as the two calls above (two launches, four
 * when the permutation runs chunked): same arguments, same outputs, same
 * bit-exactness. The fused form saves a decode step one kernel
 * boundary (the first of the two steps of the fused decode path).
 * T == 0 writes counts, offsets and padded offsets (all zero) like moe_permute.
 */
moe_status_t moe_route_permute(const float *d_logits, int T, int E, int k, int block_m,
                               int32_t *d_topk_ids, float *d_topk_w, uint32_t *d_bitmatrix,
                               int32_t *d_counts, int32_t *d_offsets, int32_t *d_padded_offsets,
                               int32_t *d_row_to_pair, int32_t *d_pair_to_row, int32_t *d_error,
                               void *stream);

/* Bytes of the prepacked weight buffer for desc (T is ignored). */
size_t moe_mxfp4_packed_bytes(const moe_layer_desc *desc);

/*
 * One-time reorder of canonical MXFP4 weights into the kernels' tile order
 * (same byte count). Canonical inputs (element 2j of a row in the low nibble
 * of byte j; one E8M0 byte per 32 consecutive K elements):
 *   d_w13_q uint8 [E, 2I, H/2], d_w13_s uint8 [E, 2I, H/32]
 *           rows [0, I) are the gate projection (W1), rows [I, 2I) the up
 *           projection (W3);
 *   d_w2_q  uint8 [E, H, I/2],  d_w2_s  uint8 [E, H, I/32].
 * d_packed must hold moe_mxfp4_packed_bytes(desc) bytes. Each 128-row tile
 * of W13 pairs 64 gate rows with their 64 up rows (the gate/up interleave of
 * txtmix.com §三). Per matrix the buffer holds the E2M1 bytes of every
 * (expert, 128-row tile, 128-element K slab) as 128 contiguous 64-byte rows,
 * then the E8M0 bytes of the same slabs, 512 per slab, in the order the
 * tensor core reads block scales from tensor memory; the GEMMs stream both
 * with TMA and never decode a weight on the SM.
 */
moe_status_t moe_mxfp4_prepack(const moe_layer_desc *desc,
                               const uint8_t *d_w13_q, const uint8_t *d_w13_s,
                               const uint8_t *d_w2_q, const uint8_t *d_w2_s,
                               void *d_packed, size_t packed_bytes, void *stream);

/*
 * Decode prepacked weights of one expert back to dense bfloat16 in canonical
 * row order (exact: every E2M1 x E8M0 product is a bfloat16 value, or an
 * infinity where it exceeds the fp32 range). Reads the same prepacked bytes
 * and scale order the GEMMs feed to the tensor core.
 *   which 0: W13, d_out uint16 (bf16 bits) [2I, H]; which 1: W2, [H, I].
 */
moe_status_t moe_mxfp4_dequant_bf16(const moe_layer_desc *desc, const void *d_packed,
                                    int which, int expert, uint16_t *d_out, void *stream);

/* Workspace bytes moe_mxfp4_forward needs for desc (all of T, H, I, E, k,
 * block_m matter). The first 4 KB hold the forward's device error word
 * (bytes 0-3) and the per-expert progress counters of the fused decode GEMMs
 * (from byte 256). */
size_t moe_mxfp4_workspace_bytes(const moe_layer_desc *desc);

/*
 * Layer output (txtmix.com §三: grouped MXFP4 expert GEMMs with fused SiLU;
 * §九: optional clamp). For token t and slot j, e = topk_ids[t, j]:
 *   gate = W1_e x_t, up = W3_e x_t           (K = H, MXFP4 weights)
 *   a = SiLU(gate) * up                      (clamped first if enabled)
 *   o = W2_e a                               (K = I)
 *   y[t] = sum_j topk_w[t, j] * o_j          (slots in ascending order)
 * Inputs:
 *   d_x              bf16 bits [T, H] row-major.
 *   d_packed         from moe_mxfp4_prepack.
 *   d_topk_w         fp32 [T, k] (from moe_route).
 *   d_offsets, d_padded_offsets, d_row_to_pair   from moe_permute.
 * Output:
 *   d_y              fp32 [T, H] (out_dtype MOE_OUT_F32) or bf16 bits [T, H]
 *                    (MOE_OUT_BF16), fully overwritten.
 * d_workspace: moe_mxfp4_workspace_bytes(desc) bytes, 256-byte aligned
 * (MOE_ERR_MISALIGNED otherwise), contents need not be initialised; the call
 * resets its device error word.
 * Numerics: block-scaled tensor-core MMAs (tcgen05 kind::mxf8f6f4) of the
 * E2M1 weights with their E8M0 scales against the activations written as sums
 * of MXFP8 terms (E4M3 values, one E8M0 scale per 32 K-elements, term scales
 * 2^-4 apart): x in 2 terms (exact for bf16 unless a 32-element block spans
 * more than 2^17), SiLU(gate)*up in 2 terms (about 8 significant bits, a bf16 h);
 * fp32 accumulation; output fp32 (or its bf16 rounding). Result within
 * 2e-2 * rms of the float64 oracle (measured errors are up to about
 * 4e-3 * rms; bf16 output adds its rounding, at most 2^-9 |y|).
 * Launches 3 to 5 kernels on `stream` (moe_mxfp4_forward_plan says which);
 * deterministic (bit-identical reruns) unless MOE_FLAG_FAST_COMBINE takes the
 * atomic combine. The GEMMs stream their weights before the kernel ahead of
 * them has finished.
 */
moe_status_t moe_mxfp4_forward(const moe_layer_desc *desc, const uint16_t *d_x,
                               const void *d_packed, const float *d_topk_w,
                               const int32_t *d_offsets, const int32_t *d_padded_offsets,
                               const int32_t *d_row_to_pair, void *d_y,
                               void *d_workspace, size_t workspace_bytes, void *stream);

/*
 * moe_mxfp4_forward with timing: identical results, plus cudaEventRecord of
 * events[0..4] (cudaEvent_t passed as void*, created by the caller on this
 * device) on `stream` before the gather, after the gather, after the W13 GEMM,
 * after the W2 GEMM and after the combine. NULL entries are skipped. With any
 * event given, the kernels run one after another without overlap, so each
 * interval is one kernel's time. Where moe_mxfp4_forward_plan reports one
 * launch for both GEMMs, a non-NULL events[2] splits them into two launches
 * (same results, bit for bit); with events[2] NULL the interval from
 * events[1] to events[3] is the fused launch.
 */
moe_status_t moe_mxfp4_forward_timed(const moe_layer_desc *desc, const uint16_t *d_x,
                                     const void *d_packed, const float *d_topk_w,
                                     const int32_t *d_offsets, const int32_t *d_padded_offsets,
                                     const int32_t *d_row_to_pair, void *d_y,
                                     void *d_workspace, size_t workspace_bytes,
                                     void *const *events, void *stream);

/* Byte offsets of the forward's intermediates inside the workspace, for
 * inspection: out[0] error word; out[1] gathered activation terms (E4M3
 * [H/128][2][R][128]: 128-element slab, term, permutation row, element);
 * out[2] their E8M0 scales as 32-bit words [H/128][2][RS] (byte b of a word:
 * 32-element block b of the slab; RS = R rounded up to 4); out[3]
 * SiLU(gate)*up terms (E4M3 [I/128][NH][R][128], NH = 2 in this build:
 * (out[4] - out[3]) / (R * I) rounded down); out[4] their scale words
 * ([I/128][NH][RS]); out[5] per-pair W2 outputs (fp32 [T*k, H]); out[6] total
 * bytes. R = moe_permute_rows_capacity(T, E, k, block_m). An element's value
 * is the sum over terms of E4M3 value * 2^(scale byte - 127). */
moe_status_t moe_mxfp4_workspace_layout(const moe_layer_desc *desc, size_t out[7]);

/*
 * What moe_mxfp4_forward launches for desc (no device work; only the shape,
 * flags and out_dtype of desc matter). out[0]: the GEMM tile regime, by
 * average rows per expert T*k/E: 0 up to 2 (weight tiles of 16 token rows),
 * 1 up to 16 (32 rows), 2 up to 64 (64 token rows: token-major tiles whose
 * two activation terms are stacked as the MMA's 128 rows against 256 weight
 * rows when H is a multiple of 256, else weight-major tiles), 3 above 64 with
 * H not a multiple of 256 (96 rows), 4 above 64 with H a multiple of 256
 * (token-major tiles of 128 rows x 256 weight rows). out[1]: 1 when W13 and W2 run as one
 * persistent launch (regime 0 with E <= 512, H and I multiples of 256 and at
 * least 512): each expert's W2 tiles start once its W13 tiles have stored
 * their h rows, tracked by per-expert counters in the workspace. out[2]: 1
 * when MOE_FLAG_FAST_COMBINE is taken (regimes 0 and 1, fp32 output).
 * out[3]: kernels launched. Returns check failures as moe_mxfp4_forward does.
 */
moe_status_t moe_mxfp4_forward_plan(const moe_layer_desc *desc, int out[4]);

/*
 * Forward without a caller workspace, for callers that cannot allocate device
 * memory where they run the layer (a runtime that forbids allocation after
 * start-up, a plugin whose host framework owns all device memory, code that
 * must not call cudaMalloc because it can synchronise the device). There is no
 * counterpart in the source pages; it is a convenience of this library.
 *   Same arguments and results as moe_mxfp4_forward, minus the workspace: the
 *   intermediates live in a static device array of MOE_NOALLOC_SCRATCH_BYTES
 *   (32 MiB) that every GPU loading this library holds until the process exits.
 *   The call allocates nothing (no cudaMalloc/cudaFree, no allocating library
 *   routine).
 *   Returns MOE_ERR_WORKSPACE when moe_mxfp4_workspace_bytes(desc) exceeds
 *   MOE_NOALLOC_SCRATCH_BYTES (e.g. H = 4096, I = 2048, E = 256, k = 6,
 *   block_m = 16 fits up to T = 25 tokens); use moe_mxfp4_forward for larger layers.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture. All calls share the array, which keeps the previous call's
 *   contents (the call clears what it needs cleared): calls whose work overlaps
 *   on the GPU, e.g. on two streams, race on it. The forward's device error
 *   word is the array's first word: read and clear it with
 *   moe_mxfp4_noalloc_read_device_error.
 */
moe_status_t moe_mxfp4_forward_noalloc(const moe_layer_desc *desc, const uint16_t *d_x,
                                       const void *d_packed, const float *d_topk_w,
                                       const int32_t *d_offsets, const int32_t *d_padded_offsets,
                                       const int32_t *d_row_to_pair, void *d_y, void *stream);

/*
 * Read and clear the device error word of moe_mxfp4_forward_noalloc on the
 * current device (the first word of its static scratch array, which host code
 * cannot name as a device pointer). Same behaviour as moe_read_device_error:
 * synchronises `stream`, writes the recorded moe_status_t value (MOE_OK if
 * none) to *code and resets the word. Allocates nothing. No counterpart in
 * the source pages.
 */
moe_status_t moe_mxfp4_noalloc_read_device_error(int *code, void *stream);

/*
 * Expert parallelism over G ranks (experts split in contiguous ranges of
 * experts_per_rank = E / G; rank g owns experts [g*EPR, (g+1)*EPR)). The layer
 * is that of txtmix.com §一 and §三; the pages run it on one GPU, so the
 * sharding has no counterpart there: the data movement below plus two
 * all-to-alls (the caller's collective library) distribute exactly the
 * single-GPU computation. A rank:
 *   1. routes and permutes its own T tokens (moe_route_permute, all E experts);
 *   2. moe_ep_dispatch_pack: send row i (i < T*k) is the bf16 activation row of
 *      the i-th pair in (expert, token) order, i.e. of pair
 *      row_to_pair[padded[e] + i - offsets[e]] for the e with
 *      offsets[e] <= i < offsets[e+1]; d_send_local_ids[i] = e % EPR. Rank g's
 *      rows are the contiguous run offsets[g*EPR] .. offsets[(g+1)*EPR].
 *      d_send_x bf16 bits [T*k, H]; d_send_local_ids int32 [T*k]. H % 8 == 0.
 *   3. exchanges the runs (all-to-all), runs moe_permute + moe_mxfp4_forward on
 *      the received rows with k = 1, E = EPR, weight 1 (the per-pair expert
 *      outputs), and sends them back (all-to-all) in the order received;
 *   4. moe_ep_combine: y[t] = sum_j topk_w[t,j] * returned[pos(t,j)] in slot
 *      order, pos(p) = offsets[e] + pair_to_row[p] - padded[e]: d_returned fp32
 *      [T*k, H] in send order, y fp32 [T, H] fully written. A pair with an id
 *      outside [0, E) or no row adds nothing and sets *d_error (nullable) to
 *      MOE_ERR_DEVICE. H % 4 == 0.
 * Both take the outputs of step 1 (offsets, padded offsets, row_to_pair or
 * pair_to_row, ids, weights) as device pointers and run on `stream`.
 */
moe_status_t moe_ep_dispatch_pack(const uint16_t *d_x, int T, int H, int E, int k, int experts_per_rank,
                                  const int32_t *d_offsets, const int32_t *d_padded_offsets,
                                  const int32_t *d_row_to_pair, uint16_t *d_send_x,
                                  int32_t *d_send_local_ids, void *stream);
moe_status_t moe_ep_combine(const float *d_returned, int T, int H, int E, int k,
                            const int32_t *d_topk_ids, const float *d_topk_w,
                            const int32_t *d_offsets, const int32_t *d_padded_offsets,
                            const int32_t *d_pair_to_row, float *d_y, int32_t *d_error, void *stream);

/*
 * Read and clear a device error word (the d_error of moe_permute or the
 * first word of a forward workspace). Synchronises `stream`. Writes the
 * recorded moe_status_t value (MOE_OK if none) to *code.
 */
moe_status_t moe_read_device_error(void *d_error_word, int *code, void *stream);

/*
 * Drop the host-side cache of TMA tensor maps (CUtensorMap, 128 bytes each).
 * moe_mxfp4_forward encodes one map per (device, buffer address, shape, box)
 * on first use and reuses it on later calls with the same buffers; the cache
 * holds at most 4096 maps and never owns or touches device memory. Call this
 * after freeing buffers that a forward used, or to return the host memory;
 * the next forward re-encodes what it needs. Thread-safe: a forward running
 * on another thread copies its maps out under the cache lock, so clearing
 * never leaves it holding a released map.
 */
void moe_clear_cache(void);

/* Number of kernels launched by this library since load (all entry points). */
uint64_t moe_launch_count(void);

/*
 * Self-test of the bounded device-side wait that every GEMM pipeline wait uses
 * (failure detection without a GPU fault). One thread waits on a
 * shared-memory mbarrier that nothing arrives on:
 *   abort_after_ns == 0: the wait gives up after limit_ns;
 *   0 < abort_after_ns < limit_ns: a second warp sets the CTA's abort flag
 *   after abort_after_ns, and the wait returns then.
 * Either way the kernel records MOE_ERR_TIMEOUT in *d_error_word (a device
 * int32, read and cleared with moe_read_device_error) and the wait's duration
 * in nanoseconds in *d_elapsed_ns (a device uint64), then exits normally.
 * limit_ns must be in (0, 1e9]; d_error_word 4-byte and d_elapsed_ns 8-byte
 * aligned. Argument errors return before the launch.
 */
moe_status_t moe_selftest_bounded_wait(uint64_t limit_ns, uint64_t abort_after_ns, int32_t *d_error_word,
                                       uint64_t *d_elapsed_ns, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_MXFP4_H */
