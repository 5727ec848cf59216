/*
 * latentmoe.h - C ABI of the LatentMoE layer forward for one GB300 (sm_103a).
 *
 * The layer (from "The Training and RL Infrastructure Behind MAI-Thinking-1",
 * section "The model the systems run", and "MAI-Base-2: Microsoft's 2.8T base
 * model, and whether its compute numbers add up", section "The model"):
 *
 *   L = x W_r^T (+ b)                       router on the full hidden state
 *   p = softmax(L); idx = stable top-k of L  (ties: lower expert index first)
 *   g[t,j] = p[t, idx[t,j]]                  (/ sum_j g if LATENTMOE_RENORM)
 *   z = x W_dn^T                             shared down-projection to the latent
 *   slots sorted by expert (counting sort, token order kept inside an expert)
 *   H = (SiLU(z W_g^T) * (z W_u^T)) W_d^T    per-expert SwiGLU on the latent
 *   c[t] = sum_j g[t,j] H[pos[t,j]]          gate-weighted combine, fp32, j order
 *   y = c W_up^T (+ (SiLU(x W_gs^T) * (x W_us^T)) W_ds^T)   up-projection + shared
 *
 * Conventions for every entry point:
 * - Return 0 (LATENTMOE_OK) on success, a negative LATENTMOE_ERR_* otherwise.
 *   No C++ exception crosses the ABI and no kernel traps.
 * - "device pointer" means memory the current CUDA device can address
 *   (cudaMalloc or a PyTorch CUDA tensor's data_ptr()). The caller owns every
 *   pointer it passes. Pointers must be 16-byte aligned.
 * - Work is enqueued on the caller's stream and returns without waiting,
 *   unless the entry says it synchronises. Launch errors are returned at
 *   once; errors found by kernels set a device status word that
 *   latentmoe_get_status reads.
 * - A handle is not thread-safe; use it from one host thread and one stream
 *   at a time. One GPU only: the handle belongs to the device that was
 *   current at latentmoe_create.
 * - Matrices are row-major in torch nn.Linear layout [out, in]; bf16 means
 *   IEEE bfloat16 stored as 16-bit words.
 */
#ifndef LATENTMOE_H
#define LATENTMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct latentmoe* latentmoe_t;
/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* latentmoe_stream_t;

/* Layer dimensions. hidden d, latent l, ffn F and shared_ffn F_s must be
 * multiples of 128 (F_s may be 0: no shared expert). 1 <= num_experts E <= 512.
 * max_tokens bounds T for every forward and sizes the workspace. */
typedef struct {
  int64_t hidden;
  int64_t latent;
  int64_t num_experts;
  int64_t ffn;
  int64_t shared_ffn;
  int64_t max_tokens;
} latentmoe_dims;

/* Device pointers to the weights, all bf16 except b_r (fp32).
 *   w_r  [E, d]        router               b_r [E] (with either bias flag)
 *   w_dn [l, d]        latent down          w_up [d, l]   latent up
 *   w_g, w_u [E, F, l] expert gate and up   w_d [E, l, F] expert down
 *   w_gs, w_us [F_s, d], w_ds [d, F_s]      shared expert (F_s > 0 only)
 * The stacked expert tensors are contiguous, expert-major. */
typedef struct {
  const void* w_r;
  const float* b_r;
  const void* w_dn;
  const void* w_g;
  const void* w_u;
  const void* w_d;
  const void* w_up;
  const void* w_gs;
  const void* w_us;
  const void* w_ds;
} latentmoe_weights;

enum {
  LATENTMOE_RENORM = 1u,      /* divide the k gates of a token by their sum */
  LATENTMOE_ROUTER_BIAS = 2u, /* add b_r to the logits (selection and softmax) */
  LATENTMOE_OUT_FP32 = 4u,    /* forward output y is fp32 instead of bf16 */
  LATENTMOE_SELECT_BIAS = 8u, /* b_r moves only the top-k choice (ranks L + b);
                                 gates stay the unbiased softmax; exported
                                 logits are unbiased. The selection-only reading
                                 of the loss-free balancer named in "The Training
                                 and RL Infrastructure Behind MAI-Thinking-1",
                                 section "Sharding and parallelism". Not together
                                 with LATENTMOE_ROUTER_BIAS. */
  LATENTMOE_FP8_EXPERTS = 16u, /* the expert GEMMs in FP8 E4M3 with delayed
                                  scaling; see "FP8 E4M3 GEMMs" below */
  LATENTMOE_FP8_DENSE = 32u    /* with LATENTMOE_FP8_EXPERTS: the latent down-
                                  and up-projections and the shared expert in
                                  FP8 E4M3 as well (the router stays fp32) */
};

enum {
  LATENTMOE_OK = 0,
  LATENTMOE_ERR_INVALID_ARG = -1,   /* NULL, T <= 0, T > max_tokens, k > E, k > 16 ... */
  LATENTMOE_ERR_UNSUPPORTED = -2,   /* dims not multiples of 128, E > 512, misaligned */
  LATENTMOE_ERR_NOT_LOADED = -3,    /* forward before latentmoe_load_weights */
  LATENTMOE_ERR_CUDA = -4,          /* a CUDA call failed; see latentmoe_last_cuda_error */
  LATENTMOE_ERR_TIMEOUT = -5,       /* a bounded device-side wait gave up */
  LATENTMOE_ERR_DEVICE_STATUS = -6, /* a kernel flagged bad data (e.g. expert id out of range) */
  LATENTMOE_ERR_OUT_OF_MEMORY = -7  /* workspace allocation failed */
};

/* Device status bits returned by latentmoe_get_status. */
enum {
  LATENTMOE_STATUS_TIMEOUT = 1u,    /* a pipeline wait in a GEMM kernel gave up */
  LATENTMOE_STATUS_BAD_EXPERT = 2u, /* an expert id outside [0, E) reached the sort */
  LATENTMOE_STATUS_ROUNDS = 4u,     /* the capacity schedule needed more rounds than
                                       max_rounds; the slots left over were not computed */
  LATENTMOE_STATUS_BOUNDS = 8u      /* bounds-checked debug build only: a store, scatter
                                       write or combine read fell outside its buffer and
                                       was skipped */
};

/* FP8 E4M3 GEMMs (LATENTMOE_FP8_EXPERTS, LATENTMOE_FP8_DENSE). "The Training and RL
 * Infrastructure Behind MAI-Thinking-1", section "2. Numerics": forward
 * GEMMs in FP8 E4M3, per-tensor scales from a 1,024-step history of absolute
 * maxima (delayed scaling). E4M3 here: 4 exponent bits (bias 7), 3 mantissa
 * bits, largest finite 448, rounding to nearest even, saturating. A tensor t
 * with scale s is stored as codes E4M3(t * (1/s)) and stands for code * s.
 * - Expert weights: latentmoe_load_weights quantizes each of W_g^e, W_u^e,
 *   W_d^e with its own scale s = max|W| / 448 (fp32), keeping the codes only
 *   (half the bytes of bf16).
 * - Activations: z (the experts' input, written by the down-projection) and
 *   h (SiLU(gate) * up) are quantized with per-tensor scales s_z, s_h. The
 *   forward uses the current scales and records max|z| and max|h|; a last
 *   kernel enters the maxima into a 1024-entry ring per tensor and sets
 *   s = max(ring) / 448 for the next forward (unchanged while the ring holds
 *   only zeros). A new handle starts with s = 1 and an empty ring.
 * - With LATENTMOE_FP8_DENSE as well: W_dn, W_up and the shared expert's
 *   W_gs, W_us, W_ds are quantized with one scale per matrix; x, the
 *   combined latent c and the shared expert's hidden SiLU(x W_gs^T) *
 *   (x W_us^T) get delayed per-tensor scales like z and h. The combine
 *   still sums in fp32 and quantizes its result; the up-projection and the
 *   shared expert's down-projection accumulate separately and are added in
 *   fp32 before the output is rounded.
 * - The router (fp32 logits from bf16 x and W_r) is never quantized; without
 *   LATENTMOE_FP8_DENSE everything outside the expert GEMMs is bf16. */
#define LATENTMOE_FP8_TENSORS 5 /* scaled activations, in order: z, h, x, c, shared hidden */

/* Create a handle on the current device: validates dims, top_k (1..16,
 * <= E) and flags, and allocates the workspace for max_tokens tokens
 * (intermediates z, h, o, c, routing metadata; about
 * max_tokens*k*(2l+F)*2 bytes). Defined by the layer statement above.
 * On error *out is left NULL and nothing stays allocated. */
int latentmoe_create(const latentmoe_dims* dims, int top_k, uint32_t flags,
                     latentmoe_t* out);

/* Load the weights (device pointers, layouts in latentmoe_weights). The
 * library copies them into memory it owns (one allocation of the weights'
 * size, freed by latentmoe_destroy or the next load) and rewrites the expert
 * weights into contiguous tiles of 128 rows x 128 bytes for its grouped
 * GEMMs (64 bf16 columns, or 128 E4M3 codes with LATENTMOE_FP8_EXPERTS;
 * the E4M3 scales and codes are computed on the device).
 * The copies and the repacking are enqueued on `stream`: the caller's
 * writes to its weight buffers must be complete, or ordered before
 * `stream`. Before returning, the call synchronises `stream` (and only
 * that stream), so the caller may free or reuse its buffers as soon as this
 * returns. Loading again on a handle frees the earlier copy first, which
 * waits for the device (cudaFree). Errors: INVALID_ARG (NULL pointer that
 * the dims or flags need), UNSUPPORTED (pointer not 16-byte aligned),
 * OUT_OF_MEMORY, CUDA. On error the handle has no weights loaded. */
int latentmoe_load_weights(latentmoe_t h, const latentmoe_weights* w,
                           latentmoe_stream_t stream);

/* The layer forward: the computation stated at the top of this file, from
 * "The Training and RL Infrastructure Behind MAI-Thinking-1", section "The
 * model the systems run" (MoE row of the shape table: softmax gating of the
 * top-k experts over the full hidden state, one shared down-projection to
 * the latent before dispatch and one up-projection after the combine,
 * SwiGLU experts on the latent; section "2. Numerics" for the fp32 router
 * logits and the fp32 combine) and "MAI-Base-2: Microsoft's 2.8T base
 * model, and whether its compute numbers add up", section "The model" (the
 * shared expert on the full width). x: device bf16 [T, d]; out: device
 * [T, d], bf16 (fp32 with LATENTMOE_OUT_FP32). 1 <= T <= max_tokens.
 * Asynchronous on `stream`;
 * no host synchronisation and no device-to-host copy happen inside.
 * out must not overlap x or the weights. Bitwise deterministic for fixed
 * inputs and device. Nothing in it synchronises the host, so it can be
 * captured into a CUDA graph once a first call outside the capture has set
 * up the kernels on the device. */
int latentmoe_forward(latentmoe_t h, const void* x, void* out, int64_t T,
                      latentmoe_stream_t stream);

/* Router replay: the forward with the expert choices given instead of
 * selected ("The Training and RL Infrastructure Behind MAI-Thinking-1":
 * the MoE layer supports router replay, section "Sharding and parallelism";
 * choices recorded at inference are replayed in the learner's pass, section
 * "4. RL infrastructure"). idx: device int32 [T, k], expert ids of each
 * token in slot order j. gates: device fp32 [T, k], or NULL to use the
 * softmax probabilities of the replayed experts under this layer's router
 * (divided by their sum with LATENTMOE_RENORM). With gates given, the router
 * GEMM is not run. Ids outside [0, E) are dropped from the combine (that slot
 * contributes nothing) and set LATENTMOE_STATUS_BAD_EXPERT. Otherwise as
 * latentmoe_forward. */
int latentmoe_forward_routed(latentmoe_t h, const void* x, const int32_t* idx,
                             const float* gates, void* out, int64_t T,
                             latentmoe_stream_t stream);

/* The same forward with HOST buffers: copies x_host (bf16 [T, d]) to the
 * device, runs latentmoe_forward, copies the result to out_host, and
 * synchronises `stream` before returning. Page-locked host memory gives
 * full copy speed; pageable memory works too. Staging buffers are allocated
 * on the first call and kept by the handle. */
int latentmoe_forward_host(latentmoe_t h, const void* x_host, void* out_host,
                           int64_t T, latentmoe_stream_t stream);

/* Pipelined form of latentmoe_forward_host for a stream of steps: enqueues
 * the copy of x_host (bf16 [T, d]) to the device, the forward on `stream`,
 * and the copy of the result to out_host, and returns without waiting. Two
 * staging slots alternate between calls, with a copy stream for each
 * direction, so the input copy of the next call and the output copy of the
 * previous one run while this call's forward does. Every call still moves
 * its own x in and its own result out. x_host must stay unchanged, and
 * out_host unread, until latentmoe_host_wait has returned; host memory must
 * be page-locked for the copies to overlap (pageable memory works but
 * serialises). A call's forward follows the earlier forwards on `stream` as
 * latentmoe_forward does; use one stream for the calls of a handle. Staging
 * slots, streams and events are made on the first call and kept by the
 * handle. Errors: as latentmoe_forward; a failed call leaves earlier calls'
 * work enqueued. */
int latentmoe_forward_host_async(latentmoe_t h, const void* x_host, void* out_host,
                                 int64_t T, latentmoe_stream_t stream);

/* Wait until every copy that latentmoe_forward_host_async enqueued (and so
 * every forward they follow) has completed. Errors: INVALID_ARG (h NULL),
 * CUDA. */
int latentmoe_host_wait(latentmoe_t h);

/* Free the workspace and the handle. NULL is accepted and ignored. */
int latentmoe_destroy(latentmoe_t h);

/* Routing from given logits (the router-replay hook and the integer parity
 * test): the softmax gating and top-k selection of "The Training and RL
 * Infrastructure Behind MAI-Thinking-1", section "The model the systems
 * run" (MoE row), with the stable ordering of its section "Bitwise
 * determinism" (equal logits: the lower expert index first), and the
 * counting sort of the slots by expert that the dropless dispatch of its
 * section "Memory and dropless MoE" works on (token order kept inside an
 * expert). From fp32 logits [T, E] (device) it computes, on `stream`,
 *   idx [T, k] int32, gates [T, k] fp32   (softmax over E, stable top-k)
 *   counts [E], offsets [E+1], perm [T*k], pos [T, k]   int32 (counting sort)
 * with the handle's k and LATENTMOE_RENORM flag. All outputs are device
 * pointers; any of counts/offsets/perm/pos may be NULL to skip the copy. */
int latentmoe_route_from_logits(latentmoe_t h, const float* logits, int64_t T,
                                int32_t* idx, float* gates, int32_t* counts,
                                int32_t* offsets, int32_t* perm, int32_t* pos,
                                latentmoe_stream_t stream);

/* Allocation-free routing. The pages have no counterpart to this entry; it
 * exists for callers that cannot allocate device memory: an application
 * whose own memory pool owns the whole device (where an extra cudaMalloc
 * fails or breaks the pool's accounting), or a latency-critical loop that
 * cannot pay for cudaFree's implicit device synchronisation.
 * It computes exactly what latentmoe_route_from_logits computes, without a
 * handle: from fp32 logits [T, E] (device), idx [T, k] int32, gates [T, k]
 * fp32, counts [E], offsets [E+1], perm [T*k] and pos [T, k] int32, all
 * device pointers supplied by the caller (none may be NULL; 4-byte aligned).
 * flags may hold only LATENTMOE_RENORM. It allocates nothing: the scratch of
 * the counting sort is one fixed device array inside the library (1 MiB plus
 * 256 bytes, held by every GPU that loads the library until the process
 * exits). Limits: 1 <= k <= 16, k <= E <= 512, and ceil(T*k / 1024) * E <=
 * 131072 (for example T*k <= 262144 at E = 512); larger sizes return
 * LATENTMOE_ERR_UNSUPPORTED before any work is enqueued.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture. The looked-up address is cached per device ordinal for the rest
 * of the process: it does not survive cudaDeviceReset (or a context other
 * than the device's primary one), after which the module is loaded anew at
 * another address; do not call this entry after resetting a device it has
 * run on. All calls share the one array and it keeps the last call's
 * contents: calls whose work overlaps on the GPU (two streams, or two host
 * threads) race and must be serialised by the caller. Asynchronous on
 * `stream`. */
int latentmoe_route_from_logits_static(const float* logits, int64_t T, int64_t E,
                                       int top_k, uint32_t flags, int32_t* idx,
                                       float* gates, int32_t* counts,
                                       int32_t* offsets, int32_t* perm, int32_t* pos,
                                       latentmoe_stream_t stream);

/* Load-balancing statistics of the last forward on this handle ("The
 * Training and RL Infrastructure Behind MAI-Thinking-1", section "Sharding
 * and parallelism": a global-batch load-balancing loss aggregated across
 * data-parallel workers and micro-batches; "Frontier Pre-training at
 * Microsoft AI", section "Reducing per-expert overhead": batched across
 * layers). The loss formula is not given, so the entry returns the
 * per-batch statistics it is built from, ready to be summed across batches,
 * ranks and layers:
 *   counts [E] int32      slots routed to each expert (sum = T*k)
 *   prob_sum [E] fp32     sum over tokens of the router's softmax
 *                         probability of each expert (sum = T)
 * Either pointer may be NULL. Device pointers; enqueued on `stream`;
 * deterministic. After a replay forward with given gates (no router run)
 * prob_sum describes the last routed forward's logits. */
int latentmoe_lbl_stats(latentmoe_t h, float* prob_sum, int32_t* counts,
                        latentmoe_stream_t stream);

/* Copy the routing state of the last forward on this handle into caller
 * device buffers (each may be NULL): logits [T, E] fp32 (bias included),
 * idx, gates, counts, offsets, perm, pos as in latentmoe_route_from_logits.
 * Enqueued on `stream`; T is the last forward's token count. */
int latentmoe_get_routing(latentmoe_t h, float* logits, int32_t* idx,
                          float* gates, int32_t* counts, int32_t* offsets,
                          int32_t* perm, int32_t* pos, latentmoe_stream_t stream);

/* Delayed-scaling state of an E4M3 handle (synchronises the device):
 * scales[LATENTMOE_FP8_TENSORS] the next forward will use, last_amax[...]
 * the maxima the last forward recorded, *steps the forwards entered. Host
 * pointers. UNSUPPORTED without LATENTMOE_FP8_EXPERTS. */
int latentmoe_get_fp8_state(latentmoe_t h, float* scales, float* last_amax,
                            int64_t* steps);

/* E4M3 codes of the last forward's z [T*k, l] and h [T*k, F] (slot order,
 * as latentmoe_get_routing's perm), copied into caller device buffers on
 * `stream`; either may be NULL. UNSUPPORTED without LATENTMOE_FP8_EXPERTS,
 * INVALID_ARG before the first forward. */
int latentmoe_get_fp8_codes(latentmoe_t h, uint8_t* z_codes, uint8_t* h_codes,
                            latentmoe_stream_t stream);

/* E4M3 codes of the last forward's x [T, d], c [T, l] and shared hidden
 * [T, F_s] (LATENTMOE_FP8_DENSE), copied into caller device buffers on
 * `stream`; any may be NULL (sh_codes must be NULL without a shared
 * expert). UNSUPPORTED without LATENTMOE_FP8_DENSE, INVALID_ARG before the
 * first forward. */
int latentmoe_get_fp8_dense_codes(latentmoe_t h, uint8_t* x_codes, uint8_t* c_codes,
                                  uint8_t* sh_codes, latentmoe_stream_t stream);

/* Set the activation scales (host [LATENTMOE_FP8_TENSORS], finite, > 0)
 * and clear the history, e.g. from a calibration run. Synchronises the
 * device. UNSUPPORTED without LATENTMOE_FP8_EXPERTS. */
int latentmoe_set_fp8_scales(latentmoe_t h, const float* scales);

/* Scales of the loaded E4M3 weights: host fp32 [3 * E + 5]: W_g, W_u, W_d
 * of each expert ([3, E]), then W_dn, W_up, W_gs, W_us, W_ds (1 where not
 * quantized). Synchronises the device. */
int latentmoe_get_fp8_weight_scales(latentmoe_t h, float* scales);

/* Quantize bf16 src [groups, rows, cols] (device, cols % 16 == 0) to E4M3
 * with one scale per group, as the expert weights are: scales[g] =
 * max|src_g| / 448 in fp32 (1 for an all-zero group), codes = E4M3(src *
 * (1/scales[g])) with the reciprocal and the product rounded to fp32 first.
 * codes: device uint8 [groups, rows, cols]; scales: device fp32 [groups].
 * No handle needed. Asynchronous on `stream`. */
int latentmoe_quantize_e4m3(const void* src, int64_t groups, int64_t rows,
                            int64_t cols, uint8_t* codes, float* scales,
                            latentmoe_stream_t stream);

/* Synchronise the device, then read and clear the device status word
 * (LATENTMOE_STATUS_* bits). Returns TIMEOUT or DEVICE_STATUS when bits
 * were set, CUDA on a CUDA error, else OK. */
int latentmoe_get_status(latentmoe_t h, uint32_t* device_status);

/* Stage timing. latentmoe_set_profiling(h, n) with n > 0 makes each forward
 * record CUDA events between its stages into one of n rotating slots
 * (forward i uses slot i % n); n = 0 turns it off. latentmoe_get_stage_times
 * synchronises on the slot's last event and writes up to `count` per-stage
 * durations in milliseconds, in the order of latentmoe_stage_name. */
int latentmoe_set_profiling(latentmoe_t h, int slots);
int latentmoe_get_stage_times(latentmoe_t h, int slot, float* ms, int count);
int latentmoe_num_stages(void);
const char* latentmoe_stage_name(int stage);

/* Multi-round fixed-capacity schedule of the expert GEMMs ("Frontier
 * Pre-training at Microsoft AI", section "Dropless MoE with tunable,
 * fixed-size memory usage"). Experts form groups of group_size consecutive
 * experts (the last may be smaller). In every round each expert first runs
 * up to `capacity` of its remaining slots; the group's unused capacity is
 * then lent to experts with slots left, lowest expert index first; an
 * expert's slots run in slot order across rounds. The rounds repeat until no
 * slot is left (the count is the same for every group), so nothing is
 * dropped and the output equals the one-pass forward. The expert hidden
 * activations h live in a fixed buffer of E * capacity rows instead of one
 * row per slot.
 * max_rounds bounds the rounds launched per forward (each launches the two
 * expert GEMMs; rounds without slots end at once); 0 chooses the worst case
 * for max_tokens (every token putting min(k, group size) slots into the
 * smallest group). Slots left after max_rounds are not computed and set
 * LATENTMOE_STATUS_ROUNDS. capacity = 0 returns to the one-pass forward.
 * Allocates the round buffer and the schedule arrays (synchronises the
 * device). Errors: INVALID_ARG (negative values, group_size outside
 * [1, E]), UNSUPPORTED (E * capacity > 2^30 rows, more than 4096 rounds),
 * OUT_OF_MEMORY. */
int latentmoe_set_capacity(latentmoe_t h, int64_t capacity, int64_t group_size,
                           int64_t max_rounds);

/* The last forward's round schedule (synchronises the device): info (host
 * int32 [3]) = {rounds the routing needed, slots left over, rounds
 * launched}; take (device int32 [rounds launched, E], may be NULL) = slots
 * of each expert in each round. UNSUPPORTED when no capacity is set. */
int latentmoe_get_rounds(latentmoe_t h, int32_t* take, int32_t* info);

/* GEMMs on SM pairs (enable = 1, the default) or on single SMs (0). The pair
 * kernels run tcgen05 MMAs with M = 256 over two SMs of a cluster.
 * - Expert GEMMs: each SM holds its weight rows and half of the token tile;
 *   used where the shapes allow (gate+up: F % 256 == 0; down: l % 512 ==
 *   0), the single-SM kernels elsewhere.
 * - Dense GEMMs (down-projection, shared expert, up-projection): pair tiles
 *   of 256 token rows, each SM holding its 128 rows and half of the weight
 *   tile.
 * Results are bitwise the same either way. Takes effect at the next forward. */
int latentmoe_set_sm_pairs(latentmoe_t h, int enable);

/* Both expert GEMMs of the one-pass forward in one launch or in two: the
 * per-expert SwiGLU FFNs of "The Training and RL Infrastructure Behind
 * MAI-Thinking-1", section "The model the systems run" (MoE row),
 * h = SiLU(z W_g^T) * (z W_u^T) then o = h W_d^T over each expert's slots.
 * The fused launch interleaves the gate+up tiles and the down tiles of the
 * SM-pair kernels in one persistent sequence: a down tile reads a feature
 * block of h once every gate+up tile of that block of its expert has stored
 * it, so the second GEMM fills the first one's tail.
 * mode 0: two launches. mode 1: one launch wherever the shapes allow it (SM
 * pairs, F % 256 == 0, l % 512 == 0, no capacity schedule). mode 2 (the
 * default): one launch where the shapes allow it and the two GEMMs have at
 * most 400 k-blocks of work per SM pair (expected from E, l, F and T k), two
 * launches otherwise (large layers, where the tails weigh little).
 * Results are bitwise the same in every mode. When the launch is fused, stage
 * "expert_gate_up" of latentmoe_get_stage_times covers both GEMMs and
 * "expert_down" is empty. Takes effect at the next forward. Errors:
 * INVALID_ARG (h NULL, mode outside [0, 2]). */
int latentmoe_set_expert_fusion(latentmoe_t h, int mode);

/* Programmatic dependent launch between the forward's kernels (enable = 1,
 * the default) or plain stream order (0). With it, each kernel's CTAs may be
 * scheduled while the kernel before it finishes and set up their shared
 * memory and TMEM meanwhile; every kernel still waits for the one before it
 * to complete before it reads that kernel's results, so the results are
 * bitwise the same either way. Takes effect at the next forward. */
int latentmoe_set_pdl(latentmoe_t h, int enable);

/* Kernel launches issued by this handle since creation. */
int latentmoe_get_launch_count(latentmoe_t h, int64_t* launches);

/* Last CUDA error code (cudaError_t value) seen by the handle, 0 if none. */
int latentmoe_last_cuda_error(latentmoe_t h);

/* Static description of a return code. */
const char* latentmoe_strerror(int code);

/* ---- Debug entry points: the tensor-core GEMM core on its own. ----------
 * C = epilogue(A B^T) for bf16 A [M, K] and B [N', K] (device, row-major).
 *   mode 0: C bf16 [M, N], B has N rows
 *   mode 1: C fp32 [M, N], B has N rows
 *   mode 2: C bf16 [M, N] = SiLU(A Bg^T) * (A Bu^T); B is [2, G*N, K]: the
 *           gate rows of all groups, then the up rows of all groups (G = 1
 *           for the dense entry, i.e. Bg = rows 0..N-1, Bu = rows N..2N-1)
 * M >= 1, K and N multiples of 128 (mode 1: N >= 1). Grouped variant: rows
 * of A and C are split by device int32 offsets [G+1] (offsets[0] = 0,
 * non-decreasing, offsets[G] <= M, G <= 512); group g multiplies with rows
 * [g*N, (g+1)*N) of B (of each half of B in mode 2). mode | 4 runs the
 * SM-pair kernel (tcgen05 cta_group::2 on clusters of two CTAs): in the
 * dense entry for every mode, in the grouped variant for modes 0 and 2
 * (N % 512 == 0 in mode 0, N % 256 == 0 in mode 2).
 * Asynchronous on `stream`; errors as above. */
int latentmoe_debug_gemm(const void* A, const void* B, void* C, int64_t M,
                         int64_t N, int64_t K, int mode,
                         latentmoe_stream_t stream);
int latentmoe_debug_grouped_gemm(const void* A, const void* B, void* C,
                                 const int32_t* offsets, int64_t groups,
                                 int64_t M, int64_t N, int64_t K, int mode,
                                 latentmoe_stream_t stream);
/* The E4M3 grouped GEMM on its own, with codes as inputs. A: codes [M, K];
 * B: codes [G*N, K] (mode 1) or [2, G*N, K] (mode 2: gate rows, then up
 * rows); scales: device fp32 [2 + G] (mode 1) or [2 + 2G] (mode 2):
 * {s_A, s_out, s_B per group (gate groups, then up groups)}.
 *   mode 1: C bf16 [M, N] = s_A s_Bg (A B_g^T) for the rows of group g
 *   mode 2: C codes [M, N] = E4M3((SiLU(s_A s_Bg A B_g^T) * (s_A s_Ug A U_g^T))
 *           / s_out); amax (device, one uint32, caller-zeroed) receives the
 *           float bits of max |h| over all rows
 * Groups as in latentmoe_debug_grouped_gemm. K and N multiples of 128.
 * mode | 4 runs the SM-pair kernel (N % 512 == 0 in mode 1, N % 256 == 0 in
 * mode 2). Synchronises `stream`. */
int latentmoe_debug_grouped_gemm_e4m3(const uint8_t* A, const uint8_t* B,
                                      const float* scales, void* C, uint32_t* amax,
                                      const int32_t* offsets, int64_t groups,
                                      int64_t M, int64_t N, int64_t K, int mode,
                                      latentmoe_stream_t stream);

/* Device status word of the debug entry points (synchronises, then clears). */
int latentmoe_debug_status(uint32_t* device_status);

/* Exercise the bounded device wait: one thread waits on an mbarrier that
 * nothing completes, gives up after limit_ns (<= 1 s) and sets
 * LATENTMOE_STATUS_TIMEOUT. Synchronises; returns LATENTMOE_ERR_TIMEOUT and
 * the status bits when the wait gave up as designed. */
int latentmoe_debug_wait_timeout(uint64_t limit_ns, uint32_t* device_status);

#ifdef __cplusplus
}
#endif

#endif /* LATENTMOE_H */
