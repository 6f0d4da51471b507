/*
 * moe_warp.h — C ABI of libmoewarp.so: one mixture-of-experts layer evaluated
 * over one speculative-decoding verification pass of n tokens, on one GB300
 * (sm_103a).
 *
 * The operation, as the sources state it:
 *   - "Deep Dive into Mixture of Experts: From 1991 to DeepSeek-V3", §2 "The
 *     Sparse-Gating Leap" (the top-k gating sketch): logits = x·W_g, keep the
 *     k largest, softmax over those k logits only, output = Σ weight·expert(x).
 *   - same post, §5 "DeepSeek-V3 and the Current State of the Art" (the routing
 *     sketch): always-on shared experts are added unweighted.
 *   - "Building a Terminal Based LLM Inference Internals Explorer - Part 3:
 *     Speculative Decoding", section "The Flow": the verifier scores the
 *     γ drafted tokens plus the bonus position in one batched call, so a
 *     verification pass holds n = γ+1 tokens.
 *   - "Speculative Decoding for Mixture-of-Experts Models: Expert Bytes, Kernel
 *     Bandwidth and the Best Draft Length", abstract: a per-slot engine reads a
 *     selected expert once per token; a deduplicating engine reads each
 *     selected expert once per pass.
 * Each expert is a SwiGLU FFN without biases:
 *   FFN_e(x) = W_down,e · ( silu(W_gate,e · x) ⊙ (W_up,e · x) ),  silu(z) = z/(1+e^−z).
 *
 * Conventions shared by every entry point
 *   - Every pointer argument except `desc`, `weights`, `u` (host structs, read
 *     during the call only) is a DEVICE pointer. The caller owns all memory;
 *     the library never allocates device memory on these paths.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream). No call synchronises the host with the device
 *     except moe_last_device_error.
 *   - Arguments are checked on the host before any launch: a bad argument
 *     returns MOE_EINVAL (nothing is launched); a shape the kernels do not
 *     cover returns MOE_EUNSUPPORTED; a launch failure returns MOE_ECUDA.
 *   - Inputs must be finite. Behaviour on NaN/Inf inputs is unspecified.
 *   - Limits: 1 ≤ n ≤ MOE_MAX_TOKENS, n·k ≤ MOE_MAX_PAIRS, 1 ≤ k ≤ E ≤
 *     MOE_MAX_EXPERTS, k ≤ MOE_MAX_TOPK, 0 ≤ s ≤ MOE_MAX_SHARED, d and I
 *     multiples of 64, every device pointer 16-byte aligned.
 */
#ifndef MOE_WARP_H
#define MOE_WARP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_MAX_TOKENS 128
#define MOE_MAX_PAIRS 512
#define MOE_MAX_EXPERTS 256
#define MOE_MAX_TOPK 16
#define MOE_MAX_SHARED 4

typedef enum {
  MOE_OK = 0,
  MOE_EINVAL = 1,       /* bad argument: null pointer, misalignment, out-of-range size */
  MOE_ECUDA = 2,        /* a CUDA runtime call failed; moe_last_cuda_error_string() says which */
  MOE_ETIMEOUT = 3,     /* a bounded device-side wait expired (reported by moe_last_device_error) */
  MOE_EUNSUPPORTED = 4, /* valid arguments that no kernel here covers */
  MOE_EDEVICE = 5       /* a kernel recorded a failed device-side check */
} moe_status;

typedef enum { MOE_W_F32 = 0, MOE_W_BF16 = 1 } moe_wdtype;

/* Shape of one MoE layer. Plain data, caller-owned. */
typedef struct {
  int32_t d;         /* model dimension (length of a hidden state x_t) */
  int32_t n_experts; /* E, routed experts */
  int32_t top_k;     /* k, experts selected per token */
  int32_t inter;     /* I, SwiGLU intermediate size of every expert (routed and shared) */
  int32_t n_shared;  /* s, always-on shared experts (0 if none) */
  int32_t wdtype;    /* moe_wdtype of the expert weights; the router W_g is always fp32 */
} moe_layer_desc;

/* Device pointers to one layer's weights, row-major, caller-owned.
 * Element type of the expert matrices is desc->wdtype (bf16 = raw 16-bit
 * bfloat16 bit patterns).                                                    */
typedef struct {
  const float* w_router; /* W_g  [E][d]     fp32: logit of expert e is Σ_i x_i·W_g[e][i] */
  const void* w_gate;    /* [E][I][d]  W_gate,e rows (output i, input d contiguous) */
  const void* w_up;      /* [E][I][d]  W_up,e */
  const void* w_down;    /* [E][d][I]  W_down,e rows (output j, input I contiguous) */
  const void* ws_gate;   /* [s][I][d]  shared experts; NULL iff s == 0 */
  const void* ws_up;     /* [s][I][d] */
  const void* ws_down;   /* [s][d][I] */
} moe_layer_weights;

/* Device outputs of moe_build_union: the union U of the experts selected in
 * one pass, and the (token, slot) pairs grouped by expert.                  */
typedef struct {
  int32_t* union_ids;   /* [E]    distinct selected experts, ascending; first *union_count valid */
  int32_t* union_count; /* [1]    |U| */
  int32_t* offsets;     /* [E+1]  pairs of union_ids[u] are rows offsets[u] .. offsets[u+1]-1 */
  int32_t* pair_tok;    /* [n*k]  token t of each pair, grouped by expert, tokens ascending */
  int32_t* pair_slot;   /* [n*k]  slot j of each pair (topk_idx[t][j] == its expert) */
  uint64_t* bytes;      /* [3]    requested expert-weight bytes of this pass:
                                  {per-slot = n·k·E_b, dedup = |U|·E_b, shared = s·E_b},
                                  E_b = 3·d·I·sizeof(weight) bytes per expert */
} moe_union;

/* Bytes of device scratch ("workspace") the engine and routing calls need
 * for passes of up to n_max tokens. 0 on invalid arguments. The workspace is
 * caller-owned, 256-byte aligned, needs no initialisation, and may be reused
 * by consecutive calls on one stream; two calls that overlap on the device
 * must not share one. For bf16 layers it includes a fixed 24 MiB region of
 * partial sums: when a pass has too few weight tiles to keep every SM busy,
 * the engine cuts each tile's reduction into pieces and adds the pieces'
 * partial sums in a fixed order (results do not depend on scheduling). It
 * also holds the count of moe_verify_pass_fused's combine.                  */
size_t moe_workspace_bytes(const moe_layer_desc* desc, int32_t n_max);

/* Gate GEMV, top-k and renormalised softmax
 * ("Deep Dive into Mixture of Experts", §2, top-k gating sketch).
 *   x        [n][d] fp32 hidden states of the pass
 *   w_router [E][d] fp32 W_g
 *   topk_idx [n][k] int32 out: the k experts with the largest logits, in
 *            descending logit order; equal logits are ordered by ascending
 *            expert index (so ties select the lower index).
 *   topk_w   [n][k] fp32 out: softmax of the k selected logits (sums to 1).
 * Logits are accumulated with a compensated (error-free-transformation) dot
 * product, so the selection agrees with an exact computation except where
 * two logits lie within ~1e-12 relative of each other.                      */
moe_status moe_route(const moe_layer_desc* desc, const float* w_router, const float* x, int32_t n,
                     int32_t* topk_idx, float* topk_w, void* workspace, size_t workspace_bytes,
                     void* stream);

/* Gate GEMV alone ("Deep Dive into Mixture of Experts", §2, top-k gating
 * sketch: the logits are x·W_g), the first step of moe_route:
 *   logits[t][e] = Σ_i x[t][i]·w_router[e][i], with the compensated dot
 *   described under moe_route.
 *   x        [n][d] fp32, 16-byte aligned;  w_router [E][d] fp32, 16-byte aligned.
 *   logits   [n][E] fp32 out (caller-owned, 4-byte aligned).
 * MOE_EINVAL for a bad descriptor, n out of range or a null or misaligned
 * pointer.                                                                  */
moe_status moe_gate(const moe_layer_desc* desc, const float* w_router, const float* x, int32_t n,
                    float* logits, void* stream);

/* Gate GEMV and top-k with a per-expert routing bias ("Deep Dive into
 * Mixture of Experts", §5, DeepSeek-style routing sketch: a bias, adjusted
 * for load balance, is added to the gate's scores before the top-k).
 *   bias     [E] fp32 device (4-byte aligned), or NULL for no bias (then the
 *            call is moe_route).
 *   bias_in_weights  1: topk_w is the softmax of the k kept biased scores,
 *            as the sketch writes it; 0: the bias only selects, and topk_w is
 *            the softmax of the kept experts' unbiased logits.
 * Selection compares fl(logit + bias[e]) (fp32 add after the compensated
 * dot); ties, order and every other argument as moe_route. MOE_EINVAL for a
 * bias_in_weights other than 0 or 1 or a misaligned bias.                  */
moe_status moe_route_biased(const moe_layer_desc* desc, const float* w_router, const float* bias,
                            int32_t bias_in_weights, const float* x, int32_t n,
                            int32_t* topk_idx, float* topk_w, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Union of the selected experts and the pairs grouped by expert
 * ("Speculative Decoding for Mixture-of-Experts Models", abstract: the
 * deduplicating engine reads each selected expert once per pass).
 *   topk_idx [n][k] as written by moe_route (values must be in [0, E)).
 *   u        device arrays sized as documented in moe_union.
 * Integer-exact; the result does not depend on thread scheduling.          */
moe_status moe_build_union(const moe_layer_desc* desc, const int32_t* topk_idx, int32_t n,
                           const moe_union* u, void* stream);

/* Routing and union in one call: the results of moe_route_biased followed by
 * moe_build_union on its topk_idx, bit for bit, in two kernel launches
 * instead of three (one CTA runs every token's top-k and then builds the
 * union from that selection without a round trip through a kernel boundary).
 *   bias, bias_in_weights  as moe_route_biased (bias NULL: plain moe_route).
 *   topk_idx, topk_w       [n][k] out, as moe_route.
 *   u                      out, as moe_build_union.
 * Argument checks and errors: those of both calls.                          */
moe_status moe_route_union(const moe_layer_desc* desc, const float* w_router, const float* bias,
                           int32_t bias_in_weights, const float* x, int32_t n,
                           int32_t* topk_idx, float* topk_w, const moe_union* u, void* workspace,
                           size_t workspace_bytes, void* stream);

/* Per-slot engine: every (token t, slot j) runs its own expert FFN, reading
 * that expert's weights for that slot alone (requested bytes n·k·E_b), and
 * every shared expert runs once over all n tokens.
 *   x        [n][d] fp32;  topk_idx/topk_w as written by moe_route.
 *   y_slot   [n][k+s][d] fp32 out: slot j < k holds topk_w[t][j]·FFN_e(x_t)
 *            with e = topk_idx[t][j]; slot k+i holds FFN_shared_i(x_t).     */
moe_status moe_verify_perslot(const moe_layer_desc* desc, const moe_layer_weights* weights,
                              const float* x, int32_t n, const int32_t* topk_idx,
                              const float* topk_w, void* workspace, size_t workspace_bytes,
                              float* y_slot, void* stream);

/* Deduplicating engine: each distinct selected expert's weights are streamed
 * from HBM once per pass and applied to every token that selected it
 * (requested bytes |U|·E_b), plus the shared experts as above.
 *   u        the moe_build_union result for the same topk_idx (read on the
 *            device only; no host synchronisation).
 *   y_slot   same layout and meaning as moe_verify_perslot.               */
moe_status moe_verify_dedup(const moe_layer_desc* desc, const moe_layer_weights* weights,
                            const float* x, int32_t n, const moe_union* u, const float* topk_w,
                            void* workspace, size_t workspace_bytes, float* y_slot,
                            void* stream);

/* Weighted combine ("Deep Dive into Mixture of Experts", §2 and §5 sketches:
 * output = shared experts + Σ weight·expert):
 *   y[t] = Σ_{j=0}^{k+s-1} y_slot[t][j]   (fixed order j = 0, 1, …; deterministic)
 *   y_slot [n][k+s][d] fp32 in;  y [n][d] fp32 out.                         */
moe_status moe_combine(const moe_layer_desc* desc, const float* y_slot, int32_t n, float* y,
                       void* stream);

/* Engines of moe_verify_pass. */
typedef enum { MOE_ENGINE_PERSLOT = 0, MOE_ENGINE_DEDUP = 1 } moe_engine;

/* One whole verification pass in one call: what moe_route_union (routing
 * with the optional bias, and the union), then moe_verify_perslot or
 * moe_verify_dedup, then moe_combine compute, on one stream, with bitwise
 * the same results as those calls made one by one. The routing kernels also
 * do the engine's prep work (its counters zeroed, x split into bf16 halves,
 * the dedup rows gathered), so the expert kernel follows them directly: four
 * kernels, one fewer than the single calls. For callers that issue passes
 * from the host one at a time (no CUDA graph), it also saves the per-call
 * host cost of three calls.
 *   weights->w_router is W_g; bias, bias_in_weights as moe_route_biased.
 *   engine   MOE_ENGINE_PERSLOT or MOE_ENGINE_DEDUP (else MOE_EINVAL).
 *   topk_idx, topk_w, u, y_slot   the intermediate outputs, written as the
 *            single calls write them (caller-owned device buffers).
 *   y        [n][d] fp32 out (16-byte aligned), as moe_combine.
 * Every argument is checked before anything is launched; the status is
 * the first failing check's, or a launch failure's.                        */
moe_status moe_verify_pass(const moe_layer_desc* desc, const moe_layer_weights* weights,
                           const float* bias, int32_t bias_in_weights, const float* x, int32_t n,
                           int32_t engine, int32_t* topk_idx, float* topk_w, const moe_union* u,
                           void* workspace, size_t workspace_bytes, float* y_slot, float* y,
                           void* stream);

/* moe_verify_pass with the weighted combine fused into the expert kernel
 * ("Deep Dive into Mixture of Experts", §2 and §5 sketches: output = shared
 * experts + Σ weight·expert): the SwiGLU product is formed in the gate/up
 * epilogue, each slot's weight is applied in the down epilogue, and the sum
 * over the k+s slots is the kernel's last phase — every CTA publishes the
 * down rows it stored with one GPU-scope release, waits (bounded) until the
 * call's rows are all stored, and sums its share of y in slot order, the
 * same additions in the same order as moe_combine. Same arguments and
 * bitwise the same outputs as moe_verify_pass, one launch fewer. Measured
 * on GB300 (DeepSeek-V2-Lite-shaped layer), a pass this way takes within
 * about 1 us of moe_verify_pass either way: the in-kernel release and wait
 * cost about what the combine launch they replace costs, which the previous
 * kernel's tail hides (programmatic dependent launch). A call whose groups are split
 * between the tensor-core and CUDA-core kernels (only when MOE_MMA_MIN_M
 * forces it) runs the combine as a launch of its own.                      */
moe_status moe_verify_pass_fused(const moe_layer_desc* desc, const moe_layer_weights* weights,
                                 const float* bias, int32_t bias_in_weights, const float* x,
                                 int32_t n, int32_t engine, int32_t* topk_idx, float* topk_w,
                                 const moe_union* u, void* workspace, size_t workspace_bytes,
                                 float* y_slot, float* y, void* stream);

/* Allocation-free variant of moe_verify_dedup (the sources have no
 * counterpart: this exists for callers, not for the method). Some callers
 * cannot allocate device memory: a plugin whose host framework owns all GPU
 * memory and hands it only input and output buffers, or a latency-critical
 * serving loop where a device allocation, with its implicit synchronisation,
 * is not allowed after start-up. This entry point takes no workspace: its
 * scratch is a fixed array of moe_noalloc_scratch_limit() bytes (32 MiB)
 * inside the library, which every GPU that loads the library keeps until the
 * process exits. It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Same arguments, outputs and numerics as moe_verify_dedup, minus the
 *     workspace. A pass whose scratch (moe_workspace_bytes(desc, n)) exceeds
 *     the limit returns MOE_EINVAL; moe_last_cuda_error_string() says why.
 *   - The first call on a device looks up the array's device address on that
 *     device (the device must be current); make that first call before any
 *     stream capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind (nothing in it needs to start at zero). Calls that overlap on
 *     the GPU — on two streams, or from two threads — race on it.
 *   - The array's address is cached per device for the life of the process,
 *     as is the device error word's: the library must not be used across a
 *     cudaDeviceReset (or any other teardown of the primary context).     */
moe_status moe_verify_dedup_noalloc(const moe_layer_desc* desc, const moe_layer_weights* weights,
                                    const float* x, int32_t n, const moe_union* u,
                                    const float* topk_w, float* y_slot, void* stream);

/* Size in bytes of the static scratch array of moe_verify_dedup_noalloc. */
size_t moe_noalloc_scratch_limit(void);

/* Failure-detection self-test (not part of the method): launches one kernel
 * that waits on a shared-memory mbarrier nothing ever arrives on, through the
 * same bounded wait every expert kernel uses, with a limit of limit_us
 * microseconds (1 .. 1,000,000) instead of the kernels' 0.4 s. The wait
 * expires, the kernel records a timeout in the device error word and
 * returns; the context stays usable. A following moe_last_device_error on
 * the same stream returns MOE_ETIMEOUT. MOE_EINVAL for a limit out of range. */
moe_status moe_diag_bounded_wait(int32_t limit_us, void* stream);

/* Synchronises `stream`, then reads and clears the library's device error
 * word: MOE_ETIMEOUT if a bounded device-side wait expired, MOE_EDEVICE if a
 * kernel recorded a failed check, MOE_ECUDA if the stream reports an error,
 * else MOE_OK.                                                             */
moe_status moe_last_device_error(void* stream);

const char* moe_status_str(moe_status s);
const char* moe_last_cuda_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_WARP_H */
