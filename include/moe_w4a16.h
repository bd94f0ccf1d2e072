/*
 * moe_w4a16 -- INT4 weight-only (W4A16) fused Mixture-of-Experts feed-forward
 * for NVIDIA GB300 (sm_103a).
 *
 * The operation (the MoE layer benchmarked on "The Commit That Captured a
 * Plateau", commit text, and "The Pivot to Real Hardware ...", Step 1 and Input
 * Knowledge items 1-2): every token t is routed to k experts e = topk_ids[t, j]
 * with weights w = topk_weights[t, j], and
 *
 *     out[t] = sum_j w * W2[e] . ( SiLU(W1g[e] . x_t) * (W1u[e] . x_t) ),
 *     SiLU(z) = z / (1 + exp(-z)),
 *
 * where W1 = [W1g; W1u] (gate rows [0, N), up rows [N, 2N)) is [2N, K] and W2 is
 * [K, N]. Weights are symmetric INT4 with one bf16 scale per group of 32 values
 * along each GEMM's reduction dimension: value = (u - 8) * scale for a stored
 * nibble u in 0..15. Activations (x, out) are bf16. The tensor cores take fp16
 * operands (kind::f16) with fp32 accumulation: the dequantised weights (u-8)*s
 * are exact in fp16 (pack rejects scales for which they would not be), every
 * token row is fed in as x * 2^-e with a power of two chosen from the row's
 * largest magnitude (exact, and undone in fp32 in the GEMM epilogues, so any
 * finite bf16 row is within range), the intermediate SiLU(g)*u is rounded once to
 * fp16 (stored as h * 2^-2e; a value that still exceeds fp16's range saturates
 * and sets MOE_W4A16_STATUS_H_SATURATED), and the output is rounded once from
 * fp32 to bf16.
 *
 * Conventions shared by every call:
 *  - Every function returns MOE_W4A16_OK (0) or a negative code; the message of
 *    the last failure on the calling thread is moe_w4a16_last_error().
 *  - Pointers documented as "device" must be device (or managed) memory of the
 *    handle's device; "host" pointers are ordinary host memory (pinned is faster).
 *  - A `stream` argument is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Calls are stream-ordered and do not synchronise the host, except
 *    where stated.
 *  - The caller owns every buffer it passes; the library never frees them.
 *  - bf16 tensors are passed as uint16_t bit patterns.
 */
#ifndef MOE_W4A16_H
#define MOE_W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MOE_W4A16_OK = 0,
  MOE_W4A16_INVALID_ARG = -1,         /* null pointer, negative size, bad handle */
  MOE_W4A16_UNSUPPORTED_SHAPE = -2,   /* K % 128, N % 128, group_size != 32, E or topk out of range */
  MOE_W4A16_WORKSPACE_TOO_SMALL = -3, /* workspace_bytes < moe_w4a16_workspace_size(h, M) */
  MOE_W4A16_CUDA_ERROR = -4,          /* a CUDA runtime call failed (message has the CUDA error) */
  MOE_W4A16_NOT_PACKED = -5,          /* forward before moe_w4a16_pack */
  MOE_W4A16_UNSUPPORTED_SCALE = -6,   /* pack: a scale outside {0} U [2^-14, 2720] in magnitude */
  MOE_W4A16_BAD_G_IDX = -7            /* pack_ex: a group index out of range, or a group whose
                                         size is not 32 */
};

/* Weight layouts accepted by moe_w4a16_pack_ex. */
enum {
  MOE_W4A16_LAYOUT_GPTQ = 0,              /* codes [R/8, C] int32, scales [R/32, C] per expert */
  MOE_W4A16_LAYOUT_COMPRESSED_TENSORS = 1 /* codes [C, R/8] int32, scales [C, R/32] per expert */
};

/* Device status bits (see moe_w4a16_status). */
enum {
  MOE_W4A16_STATUS_BAD_EXPERT_ID = 1, /* a topk_ids entry was outside [0, E); that slot was skipped */
  MOE_W4A16_STATUS_TIMEOUT = 2,       /* a pipeline wait in a GEMM kernel gave up; output is invalid */
  MOE_W4A16_STATUS_H_SATURATED = 4,   /* an intermediate activation exceeded fp16's range and was
                                         saturated to +-65504; the output is inexact */
  MOE_W4A16_STATUS_BAD_SCHEDULE = 16  /* malformed stream-K boundaries were ignored (the GEMMs split
                                         their steps evenly instead); the output is still correct */
};

typedef struct moe_w4a16_ctx* moe_w4a16_t;

/* Create a handle for E experts, hidden size K, intermediate size N, top-k
 * routing and INT4 group size (must be 32). Binds to the current CUDA device and
 * allocates the packed weight storage there (cudaMalloc, same byte count as the
 * GPTQ-style inputs: E*(3*N*K/2 + 2*(2N*K/32 + K*N/32)) bytes).
 * Requirements: K % 128 == 0, N % 128 == 0, 1 <= E <= 1024, 1 <= topk <= E.
 * Host-synchronous. */
int moe_w4a16_create(int E, int K, int N, int topk, int group_size, moe_w4a16_t* out);

/* Free the packed weights and the handle. Synchronises the device first. */
int moe_w4a16_destroy(moe_w4a16_t h);

/* Repack GPTQ-style weights into the library's device layout ("The Pivot to
 * Real Hardware ...", Step 2: GPTQ int32 in, hardware-friendly tiles out, no
 * act-order permutation). All four inputs are device pointers, C-contiguous:
 *   w1_q int32 [E, K/8, 2N]   code i of a word = element 8*row+i (bits 4i..4i+3)
 *   w1_s bf16  [E, K/32, 2N]
 *   w2_q int32 [E, N/8, K]
 *   w2_s bf16  [E, N/32, K]
 * Every scale must be 0 or have a finite magnitude in [2^-14, 2720], the range in
 * which each dequantised weight (u - 8) * s, and the dequantisation's offset
 * term -24 * s, are exact fp16 numbers (a practical GPTQ scale is far below the
 * ceiling: |w| <= 8 * s); otherwise
 * the call returns MOE_W4A16_UNSUPPORTED_SCALE and the handle stays unpacked.
 * Synchronises `stream` (to read the scale check); the inputs may be freed once
 * it returns. */
int moe_w4a16_pack(moe_w4a16_t h, const int32_t* w1_q, const uint16_t* w1_s,
                   const int32_t* w2_q, const uint16_t* w2_s, void* stream);

/* moe_w4a16_pack with a choice of input layout and optional act-order group
 * indices. Sources: "The Pivot to Real Hardware ...", The Context: Where We
 * Stand (the model's INT4 weights ship in the compressed-tensors format) and
 * Step 2: The Repack Pipeline (the repack takes GPTQ weights plus a
 * permutation, empty when the model was quantised without activation order).
 * Per expert, with R the reduction length and C the output features of a matrix
 * (w1: R = K, C = 2N, gate features first; w2: R = N, C = K):
 *   layout MOE_W4A16_LAYOUT_GPTQ: codes [R/8, C], scales [R/32, C] (as pack);
 *   layout MOE_W4A16_LAYOUT_COMPRESSED_TENSORS: codes [C, R/8] (every output
 *     feature's row contiguous, code i of word [c, r] = element 8r+i in bits
 *     4i..4i+3, the stored nibble u standing for u - 8), scales [C, R/32].
 * w1_g_idx / w2_g_idx (int32 [E, K] / [E, N], device, or NULL for none): the
 * act-order group of every reduction element -- element r of a matrix uses the
 * scale of group g_idx[r] instead of r / 32. Every group must hold exactly 32
 * elements, else MOE_W4A16_BAD_G_IDX. The library packs each matrix's elements
 * in group order (a stable sort by group); the forward then gathers the hidden
 * states of w1's experts in that order and w1's output features are stored in
 * w2's order, so the results are those of the unpermuted weights (to rounding)
 * at no extra cost in the GEMMs. With act-order the handle keeps the packing
 * order on the device (4 * E * (K or N) bytes per matrix), and the intermediate
 * returned by moe_w4a16_read_intermediate is in w2's packing order.
 * Same checks, synchronisation and ownership as moe_w4a16_pack. */
int moe_w4a16_pack_ex(moe_w4a16_t h, const int32_t* w1_q, const uint16_t* w1_s,
                      const int32_t* w2_q, const uint16_t* w2_s, int layout,
                      const int32_t* w1_g_idx, const int32_t* w2_g_idx, void* stream);

/* Bytes of device workspace that moe_w4a16_forward needs for M tokens (and any
 * smaller M) with the handle's current grid size (MOE_W4A16_OPT_NUM_CTAS: a pair
 * of split-K partial tiles per CTA). Holds the per-call routing tables, the
 * expert-sorted activations, the intermediate activations, split-K partial
 * tiles and the fp32 output accumulator. No state persists in it between calls. */
size_t moe_w4a16_workspace_size(moe_w4a16_t h, int M);

/* The fused forward. Device pointers:
 *   hidden       bf16  [M, K]
 *   topk_ids     int32 [M, topk]   expert ids; entries outside [0, E) are skipped
 *                                  and set MOE_W4A16_STATUS_BAD_EXPERT_ID
 *   topk_weights fp32  [M, topk]
 *   out          bf16  [M, K]      written completely (rounded to nearest even)
 *   workspace    >= moe_w4a16_workspace_size(h, M) bytes, 256-byte aligned
 * M == 0 is a no-op. Launches 5 kernels on `stream` (4 when M * topk <= 32:
 * routing + gather in one; 3 with MOE_W4A16_OPT_FUSED_SMALL_BATCH),
 * allocates nothing and makes no host-synchronising call, so it may be captured
 * into a CUDA graph and replayed with new inputs in the same buffers. */
int moe_w4a16_forward(moe_w4a16_t h, const uint16_t* hidden, const int32_t* topk_ids,
                      const float* topk_weights, uint16_t* out, int M,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Router ("The Weight-Streaming Threshold", Input Knowledge Required: the gating
 * network picks the k experts a token is sent to; the workloads route by
 * "router logits -> softmax top-k, renormalised"). Device pointers:
 *   router_logits fp32  [M, E]
 *   topk_ids      int32 [M, topk]  out: the k largest logits' experts, in
 *                                  descending order, equal logits by ascending id
 *   topk_weights  fp32  [M, topk]  out: softmax over all E restricted to those k
 *                                  and renormalised, exp(l_j - l_0) / sum_i exp(l_i - l_0)
 * 1 <= topk <= min(E, 32), E <= 1024. Logits should be finite (a NaN ranks as
 * -infinity). One launch on `stream`, no host synchronisation. */
int moe_w4a16_route(const float* router_logits, int M, int E, int topk, int32_t* topk_ids,
                    float* topk_weights, void* stream);

/* moe_w4a16_forward with the router in front: routes router_logits fp32 [M, E]
 * (as moe_w4a16_route, topk <= 32), writes topk_ids / topk_weights (device
 * outputs, [M, topk]) and runs the forward on them. For M * topk <= 32 the
 * routing runs inside the forward's first launch (4 launches in all); otherwise
 * a router launch precedes the forward's 5. Same workspace as moe_w4a16_forward. */
int moe_w4a16_forward_logits(moe_w4a16_t h, const uint16_t* hidden, const float* router_logits,
                             int32_t* topk_ids, float* topk_weights, uint16_t* out, int M,
                             void* workspace, size_t workspace_bytes, void* stream);

/* End-to-end variant with HOST buffers (same shapes as moe_w4a16_forward); it
 * synchronises `stream` before returning, so the buffers may be reused at once.
 * Batches whose hidden states take at most 1 MiB are zero-copy: when all four
 * buffers are pinned host memory (page-locked or registered; hidden and out
 * 16-byte aligned) the kernels read the inputs and write `out` in place over the
 * host-device link; pageable buffers are first copied into a pinned staging block
 * the handle allocates on first use (kept until moe_w4a16_destroy) and read from
 * there. Larger batches are copied host->device into the workspace, and `out`
 * back, by the copy engines. The workspace must hold
 * moe_w4a16_workspace_size(h, M) + moe_w4a16_host_staging_size(h, M) bytes
 * whichever route is taken. Not safe to call on one handle from two threads at
 * once (the staging block is shared). */
size_t moe_w4a16_host_staging_size(moe_w4a16_t h, int M);
int moe_w4a16_forward_host(moe_w4a16_t h, const uint16_t* hidden, const int32_t* topk_ids,
                           const float* topk_weights, uint16_t* out, int M,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Expert parallelism ("The Weight-Streaming Threshold", Assumptions Embedded in
 * the Analysis: with TP-8 each GPU holds a subset of the experts and an
 * AllReduce combines the GPUs' outputs). A layer of E_total experts is split
 * into contiguous ranges; each part is a handle of its own:
 *
 * moe_w4a16_create_ep: a handle holding experts [expert_begin, expert_end) of
 * E_total (0 <= expert_begin < expert_end <= E_total <= 1024, 1 <= topk <=
 * E_total; other requirements and allocation as moe_w4a16_create with E =
 * expert_end - expert_begin). moe_w4a16_pack / pack_ex then take the local
 * experts' weights only ([expert_end - expert_begin, ...]). The forward calls take
 * the layer's expert ids: a slot routed to an expert outside the range is
 * skipped silently (another part holds it); an id outside [0, E_total) still
 * sets MOE_W4A16_STATUS_BAD_EXPERT_ID. The router variant routes over all
 * E_total logits ([M, E_total]).
 *
 * moe_w4a16_forward_partial: the forward without the output rounding: writes
 * partial fp32 [M, K] (device, 16-byte aligned, overwritten) = the weighted sum
 * over this handle's experts only. Launches on `stream` as moe_w4a16_forward,
 * with no finalize step. Summing the parts' partials (an all-reduce across the
 * ranks) and rounding the sum with moe_w4a16_finalize gives the full layer's
 * output, up to the order of the fp32 additions.
 *
 * moe_w4a16_finalize: out bf16 [n] = round-to-nearest-even of acc fp32 [n]
 * (device, 16-byte aligned, n a multiple of 8). One launch on `stream`. */
int moe_w4a16_create_ep(int E_total, int expert_begin, int expert_end, int K, int N, int topk,
                        int group_size, moe_w4a16_t* out);
int moe_w4a16_forward_partial(moe_w4a16_t h, const uint16_t* hidden, const int32_t* topk_ids,
                              const float* topk_weights, float* partial, int M,
                              void* workspace, size_t workspace_bytes, void* stream);
int moe_w4a16_finalize(const float* acc, uint16_t* out, long long n, void* stream);

/* Read the device status word of the last forward that used `workspace`
 * (bits MOE_W4A16_STATUS_*; 0 = clean). Synchronises `stream`. */
int moe_w4a16_status(moe_w4a16_t h, const void* workspace, int32_t* status, void* stream);

/* Thread-local text of the last error (never NULL). */
const char* moe_w4a16_last_error(void);

/* Tuning and measurement knobs.
 *   MOE_W4A16_OPT_NUM_CTAS   persistent GEMM grid size (default: SM count; 1..256)
 *   MOE_W4A16_OPT_PROFILE    1 = record CUDA events between the forward's kernels
 *                            (read with moe_w4a16_kernel_times; perturbs overlap)
 *   MOE_W4A16_OPT_PDL        1 = launch dependent kernels with programmatic
 *                            dependent launch (default 1)
 *   MOE_W4A16_OPT_STEP_COST_GATEUP, MOE_W4A16_OPT_STEP_COST_DOWN
 *                            stream-K balance of each GEMM for batches with
 *                            M * topk > 32: a pipeline step whose token tile has
 *                            ng row groups of 16 counts as 8 + value * max(0, ng - 2);
 *                            0 = split the steps evenly (range 0..64)
 *   MOE_W4A16_OPT_WAIT_LIMIT_US
 *                            longest time a GEMM pipeline wait may take before the
 *                            kernel gives up, sets MOE_W4A16_STATUS_TIMEOUT, lets
 *                            its in-flight copies and MMAs land and returns: value
 *                            microseconds at clocks up to 4 GHz, counted in SM
 *                            cycles (0 = the default, about 4 s at 2 GHz). The
 *                            output of a call that gave up is invalid; the next
 *                            call is not affected.
 *   MOE_W4A16_OPT_TEST_WAIT_NEVER_COMPLETES
 *                            test hook: 1 makes each GEMM's epilogue first wait on
 *                            a barrier nothing arrives on, so that the give-up path
 *                            above runs (use with a short wait limit). 0 = off.
 *   MOE_W4A16_OPT_FUSED_SMALL_BATCH
 *                            1 = a forward with M * topk <= 32 whose ids are given
 *                            runs both GEMMs in one cooperative launch (the down
 *                            GEMM's weights stream while the gate/up GEMM
 *                            finishes); 0 (default) = two launches. Either way the
 *                            same arithmetic.
 *   MOE_W4A16_OPT_GEMV_SMALL_BATCH
 *                            where a forward (the fused launch off) computes its two
 *                            expert products on the CUDA cores instead of the
 *                            tensor cores: 1 (default) and 3 = batches of
 *                            M * topk <= 256 routed slots (on GB300 faster than
 *                            the tensor cores there with top-8 of 384 experts);
 *                            2 = single tokens (M == 1) only; 0 = never. The
 *                            CUDA-core kernels compute matrix-vector products over
 *                            tiles of at most 4 token rows per expert: activations
 *                            as 16-bit block fixed point per scale group of 32
 *                            (a power-of-two exponent each), products with the
 *                            4-bit codes summed exactly in int32 (dp2a), the -8
 *                            offset applied through the group's exact value sum,
 *                            one fp32 rounding per group. The tensor-core kernels
 *                            round the activations to fp16 instead; the two agree
 *                            to about 2^-12 of the output's magnitude.
 *   MOE_W4A16_OPT_GEMV_ONE_LAUNCH
 *                            1 = with at most 32 routed slots on the CUDA cores and
 *                            a grid of at most one CTA per SM, both products run in
 *                            one cooperative launch (the down product's weights
 *                            stream right after the gate/up product's; its
 *                            activation rows are taken over from the gate/up
 *                            epilogues of the whole grid through counters);
 *                            0 (default) = two launches, measured faster on GB300
 *                            (the cooperative launch cannot start while the
 *                            routing kernel runs). Same arithmetic. */
enum { MOE_W4A16_OPT_NUM_CTAS = 1, MOE_W4A16_OPT_PROFILE = 2, MOE_W4A16_OPT_PDL = 3,
       MOE_W4A16_OPT_STEP_COST_GATEUP = 4, MOE_W4A16_OPT_STEP_COST_DOWN = 5,
       MOE_W4A16_OPT_WAIT_LIMIT_US = 6, MOE_W4A16_OPT_TEST_WAIT_NEVER_COMPLETES = 7,
       MOE_W4A16_OPT_FUSED_SMALL_BATCH = 8, MOE_W4A16_OPT_GEMV_SMALL_BATCH = 9,
       MOE_W4A16_OPT_GEMV_ONE_LAUNCH = 10 };
int moe_w4a16_set_option(moe_w4a16_t h, int option, int value);

/* Milliseconds of each kernel of the last profiled forward, in launch order
 * (align, gather, gemm1, gemm2, finalize); when M * topk <= 32 the routing and
 * the gather run as one kernel, reported as align (gather then reads ~0), and the
 * down GEMM rounds the output itself (finalize then reads ~0).
 * Synchronises on the recorded events.
 * `n` is the capacity of `ms`; returns the number written or a negative code. */
int moe_w4a16_kernel_times(moe_w4a16_t h, float* ms, int n);

/* Total packed weight bytes held by the handle (weights + scales). */
size_t moe_w4a16_packed_bytes(moe_w4a16_t h);

/* ---- test-only exports ------------------------------------------------- */

/* Token->expert align on its own, for bit-exact checks. Device pointers:
 * topk_ids int32 [M, topk]; sorted_ids int32 [capacity]; expert_offsets int32
 * [E+1]; num_padded int32 [1]. For every expert in id order: the flat slot ids
 * t*topk+j routed to it in ascending order, then the sentinel M*topk up to a
 * multiple of `block`. capacity must be >= M*topk + min(E, M*topk)*(block-1). */
int moe_w4a16_align_debug(const int32_t* topk_ids, int M, int topk, int E, int block,
                          int32_t* sorted_ids, int32_t* expert_offsets, int32_t* num_padded,
                          int capacity, void* stream);

/* Invert the repack: write the handle's packed weights back in the layout and
 * order they were packed from (moe_w4a16_pack or moe_w4a16_pack_ex: device
 * pointers, the same shapes; codes and scales bit for bit). */
int moe_w4a16_unpack_debug(moe_w4a16_t h, int32_t* w1_q, uint16_t* w1_s,
                           int32_t* w2_q, uint16_t* w2_s, void* stream);

/* Copy the intermediate activations SiLU(gate)*up of the last forward that used
 * `workspace` into h_rows fp32 [M*topk, N] (device), row = flat slot id
 * t*topk+j: the fp16 tensor-core operand with the row's prescale undone; rows of
 * skipped slots are left untouched. With act-order on w2 the features come in
 * w2's packing order (see moe_w4a16_pack_ex). */
int moe_w4a16_read_intermediate(moe_w4a16_t h, const void* workspace, int M,
                                float* h_rows, void* stream);

/* Copy the fp32 accumulator of the last forward that used `workspace` (with M
 * tokens) -- sum_j w * W2[e] . h before the output's rounding to bf16 -- into acc
 * fp32 [M, K] (device). */
int moe_w4a16_read_accumulator(moe_w4a16_t h, const void* workspace, int M, float* acc,
                               void* stream);

/* Copy the stream-K boundaries of the last forward that used `workspace` (with M
 * tokens) to host memory: bounds[w * (G + 1) + c] = first pipeline step of CTA c
 * in GEMM w (0 gate/up, 1 down), G = the grid size (MOE_W4A16_OPT_NUM_CTAS);
 * *flags = bit w set when GEMM w used those boundaries (else it split its steps
 * evenly and the table is stale). `n` is the capacity of `bounds`. Synchronises
 * `stream`; returns the number of entries written or a negative code. */
int moe_w4a16_schedule_debug(moe_w4a16_t h, const void* workspace, int M, int64_t* bounds,
                             int n, int* flags, void* stream);

/* ---- allocation-free variant ------------------------------------------ */

/* The benchmark pages have no counterpart of this call; it exists for callers
 * that cannot allocate device memory -- code running where cudaMalloc is not
 * allowed or not wanted (inside a memory-pool-owning runtime, after device memory
 * has been committed to a fixed budget, or in a plug-in that must not touch the
 * host application's allocator) and so cannot provide the workspace that
 * moe_w4a16_forward needs.
 *
 * Same computation, arguments and device pointers as moe_w4a16_forward, minus the
 * workspace: the scratch lives in a fixed 48 MiB array in the library's device
 * image (MOE_W4A16_NOALLOC_WORKSPACE_BYTES), present on every GPU that loads the
 * library until the process exits. Calls whose moe_w4a16_workspace_size(h, M)
 * exceeds it are rejected with MOE_W4A16_WORKSPACE_TOO_SMALL and a message giving
 * both sizes (at E=384, K=7168, N=2048, top-8 and the default grid this admits
 * M <= 16 tokens).
 * The first call on a device looks up the array's device address (a one-time
 * set-up per device, repeated automatically if the device's context has been
 * re-created since, e.g. after cudaDeviceReset); make that first call before any
 * stream capture.
 * Every call on a device shares the one array: calls that can overlap on the GPU
 * (different streams without ordering between them) race and give wrong results;
 * calls ordered on one stream are safe. Each call re-initialises what the
 * forward needs zeroed, so leftovers of an earlier call do not matter.
 * No cudaMalloc, cudaFree or other allocating routine is called. */
#define MOE_W4A16_NOALLOC_WORKSPACE_BYTES (48u << 20)
int moe_w4a16_forward_noalloc(moe_w4a16_t h, const uint16_t* hidden, const int32_t* topk_ids,
                              const float* topk_weights, uint16_t* out, int M, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_W4A16_H */
