/*
 * moe_ffn.h -- C ABI of the MoE FFN layer forward for GB300 (sm_103a).
 *
 * The layer (one tensor-parallel rank, one GPU):
 *
 *   out[t] = sum_j w[t,j] * E_{id[t,j]}(x[t]) + S(x[t])
 *   E_e(v) = ( SiLU(v . Wg_e^T) * (v . Wu_e^T) ) . Wd_e^T      (routed expert e)
 *   S(v)   = ( SiLU(v . Wsg^T)  * (v . Wsu^T)  ) . Wsd^T       (shared expert)
 *
 * id[t,:] are the k experts with the largest fp32 router logits
 * l[t,e] = x[t] . Wr[e] + b[e], and w[t,:] is the softmax over those k logits.
 *
 * Source of the structure: "Ascend 910C LLM inference optimisation, part 2"
 * (Dewu Tech), section on MoE multi-stream overlap -- the layer runs the routed
 * experts (GroupedMatmul), the shared expert and a reduction; the shared
 * expert's gate_up (part 1) and down (part 2) matmuls read the same hidden
 * states and do not depend on the routed path, so they run on a side stream
 * that the default stream waits for; the routed path is dispatch -> gmm1 ->
 * gmm2 -> combine.  The reduction is the identity at one rank.  The router,
 * the top-k renormalisation and SiLU*mul follow the layer's definition in the
 * benchmark shapes (fp32 router, renormalised top-k softmax, bf16 SwiGLU).
 *
 * Conventions for every call:
 *  - Pointers are DEVICE pointers unless stated otherwise; the caller owns all
 *    memory, streams and events.  No call allocates device memory.  The
 *    matmul operands (a, w and out of the grouped matmul; x, out, the
 *    workspace and the expert weights of the layer forward) must be device
 *    memory of the current device (cudaMalloc-type memory, not host, managed
 *    or another GPU's memory): the kernels read them with TMA, some of it
 *    multicast between the two CTAs of a cluster of this GPU.  Other
 *    pointers are refused with MOE_ERR_UNSUPPORTED before any launch.  The
 *    library runs on one GPU: it makes no peer access and no collective.
 *  - Every call is asynchronous on the given stream and never synchronises
 *    with the host (moe_last_device_error excepted).
 *  - bf16 tensors are row-major, 16-byte aligned; K-major weights ([rows][K]).
 *  - Arguments are checked on the host before anything is launched:
 *    MOE_ERR_INVALID for null/negative/inconsistent arguments,
 *    MOE_ERR_UNSUPPORTED for shapes or alignments the kernels do not handle
 *    (there is no fallback path), MOE_ERR_WORKSPACE for a workspace that is too
 *    small, MOE_ERR_CUDA if a launch fails.
 *  - Device-side checks (an expert id out of range, group offsets that are not
 *    monotone or exceed the stated row bound, a bounded wait that expired)
 *    skip the offending work and record the first such code in a per-device
 *    status word read by moe_last_device_error().
 *  - T == 0 is valid and launches nothing.
 */
#ifndef MOE_FFN_H_
#define MOE_FFN_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID = -1,
  MOE_ERR_UNSUPPORTED = -2,
  MOE_ERR_WORKSPACE = -3,
  MOE_ERR_CUDA = -4,
  MOE_ERR_TIMEOUT = -5,      /* device: a bounded wait expired */
  MOE_ERR_DEVICE_CHECK = -6  /* device: an index or offset failed its range check */
} moe_status;

/* Layer sizes: hidden H, routed experts E, top-k k, expert intermediate I,
 * shared-expert intermediate I_s (0 = no shared expert). */
typedef struct {
  int H, E, k, I, I_s;
} moe_dims;

/* Layer weights (device pointers, caller-owned).
 *  w_router    fp32 [E][H]
 *  router_bias fp32 [E] or NULL; -INFINITY keeps an expert from being chosen
 *  w_gate_up   bf16 [E][2I][H]: rows 0..I-1 gate, rows I..2I-1 up
 *  w_down      bf16 [E][H][I]
 *  ws_gate_up  bf16 [2I_s][H] (NULL iff I_s == 0)
 *  ws_down     bf16 [H][I_s]  (NULL iff I_s == 0) */
typedef struct {
  const float* w_router;
  const float* router_bias;
  const void* w_gate_up;
  const void* w_down;
  const void* ws_gate_up;
  const void* ws_down;
} moe_weights;

/* Router: fp32 logits l[t,e] = sum_h x[t,h]*Wr[e,h] + b[e]; the k largest
 * (ties to the lower id) become topk_ids[t,:] in ascending id order and
 * topk_w[t,:] = softmax over those k logits (the full softmax over E
 * renormalised over the chosen k).
 *  x        bf16 [T][H];  w_router fp32 [E][H];  bias fp32 [E] or NULL
 *  topk_ids int32 [T][k] (out);  topk_w fp32 [T][k] (out)
 *  ws       scratch of moe_route_workspace_bytes(T, H, E) bytes (16-byte aligned)
 * From T = 512 tokens (E and H multiples of 64) the logits are computed on the
 * tensor cores from an exact three-term bf16 split of the fp32 weights, with
 * fp32 accumulation; below that, with fp32 FMAs.  Either way the logits carry
 * fp32 accuracy; expert choices whose logits differ by less than the fp32
 * summation error can differ from another fp32 evaluation order.
 * Supported: 1 <= k <= min(E, 16), E <= 512, H % 8 == 0. */
MOE_API size_t moe_route_workspace_bytes(int T, int H, int E);
MOE_API int moe_route(const void* x, const float* w_router, const float* bias, int T, int H, int E, int k,
              int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Dispatch (permute): a deterministic counting sort of the T*k (token, slot)
 * pairs by (expert ascending, token ascending).
 *  topk_ids       int32 [T][k], distinct ids in [0,E) per token (device-checked)
 *  expert_offsets int32 [E+1] (out): exclusive prefix sum of per-expert counts
 *  sorted_token   int32 [T*k] (out): token of permuted row r
 *  inv_perm       int32 [T*k] (out): permuted row of pair (t,j) at t*k+j
 *  x, x_perm      bf16 [T][H] in, bf16 [T*k][H] out (x_perm[r] = x[sorted_token[r]]);
 *                 x_perm may be NULL to skip the row gather (x is then unused)
 *  ws             scratch of moe_permute_workspace_bytes(T, E) bytes
 * Bit-exact: the result does not depend on thread scheduling. */
MOE_API size_t moe_permute_workspace_bytes(int T, int E);
MOE_API int moe_permute(const int32_t* topk_ids, const void* x, int T, int H, int E, int k, int32_t* expert_offsets,
                int32_t* sorted_token, int32_t* inv_perm, void* x_perm, void* ws, size_t ws_bytes,
                cudaStream_t stream);

/* GroupedMatmul (gmm1/gmm2): for each group g, rows r in
 * [group_offsets[g], group_offsets[g+1]) of A:
 *   act == 0:  out[r, :] = A[r, :] . W[g]^T                  W bf16 [G][N][K]
 *   act == 1:  out[r, :] = SiLU(A[r] . Wg^T) * (A[r] . Wu^T)  W bf16 [G][2N][K]
 *              (rows 0..N-1 of W[g] gate, N..2N-1 up)
 *  a             bf16 [rows_max][K]
 *  group_offsets int32 [G+1] on the device (never read by the host); NULL
 *                means one group covering rows [0, rows_max) (requires G == 1)
 *  rows_max      host upper bound on group_offsets[G] (device-checked)
 *  out           bf16 [rows_max][N]; rows outside every group are not written
 *  ws            split-K scratch of moe_grouped_gemm_workspace_bytes(...) bytes,
 *                256-byte aligned, or NULL (no split-K).  It must be zero-filled
 *                before its first use; every call leaves its counters zero
 *                again (after a device error, zero it again).  The counters
 *                fill the first 64 KiB whatever the shape, so calls of any
 *                shapes may use one buffer in turn (sized for the largest).
 *                Calls that share a scratch buffer must not overlap on the GPU.
 * bf16 inputs, fp32 accumulation (in tensor memory; on the CUDA cores when
 * rows_max is 1, a pure weight stream), bf16 (round-to-nearest) output.  With
 * scratch, launches whose groups have at most 16 rows may cut a unit's K range
 * between CTAs (S-way split or stream-K); the partial sums are added in a
 * fixed order, so results do not depend on scheduling.
 * Supported: K % 64 == 0, N % 64 == 0, G <= 1024. */
MOE_API size_t moe_grouped_gemm_workspace_bytes(int G, int rows_max, int N, int K, int act);
MOE_API int moe_grouped_gemm(const void* a, const void* w, const int32_t* group_offsets, int G, int rows_max, int N,
                             int K, int act, void* out, void* ws, size_t ws_bytes, cudaStream_t stream);

/* moe_grouped_gemm for callers that cannot allocate device memory: for
 * example code that runs inside another runtime's execution step, where a
 * cudaMalloc is forbidden or would stall the stream, or that must leave every
 * device allocation to an allocator it does not own.  Same arguments, result
 * and checks as moe_grouped_gemm, without the ws/ws_bytes pair: the split-K
 * scratch is a fixed array of MOE_NOALLOC_SCRATCH_BYTES in the library's own
 * device memory, held on every GPU that loads the library until the process
 * exits.  The pages describe no such call; it is an addition of this library.
 *  - Allocates nothing: no cudaMalloc or cudaFree, no allocating library call.
 *    It clears the scratch counters with cudaMemsetAsync on `stream`.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress with that device current) and keeps it for that
 *    device's current context; make that first call before any stream
 *    capture on the device.  A call in a new context (after cudaDeviceReset,
 *    say) looks the address up again, so again call it once before capturing.
 *  - Every call uses the same array and it keeps the previous call's data:
 *    calls that overlap on the GPU (other streams, other threads) race on it
 *    and give wrong results.  Order them on one stream.
 *  - A launch uses at most a 64 KiB counter region plus 1024 partial slots of
 *    at most 16 KiB, so every supported shape fits the array (the call checks
 *    this and would return MOE_ERR_WORKSPACE). */
#define MOE_NOALLOC_SCRATCH_BYTES (24u << 20)
MOE_API int moe_grouped_gemm_noalloc(const void* a, const void* w, const int32_t* group_offsets, int G, int rows_max,
                                     int N, int K, int act, void* out, cudaStream_t stream);

/* GroupedMatmul with FP8 weights (the w8a8_dynamic matmul configuration of the
 * xLLM PR "FlashComm1 + matmul-reduce-scatter", configuration section, taken
 * for the weight side; activations stay bf16): W holds e4m3 codes (OCP 8-bit
 * float: sign, 4 exponent bits with bias 7, 3 mantissa bits; the NaN codes
 * 0x7f/0xff are not valid weights) with one fp32 scale per weight row, and the
 * product uses W[g][n][k] = e4m3(code) * w_scale[g][n]:
 *   act == 0:  out[r, n] = s[g][n] * (A[r] . code[g][n])          w  [G][N][K]
 *   act == 1:  out[r, n] = SiLU(s_g * A[r].Wg[n]) * (s_u * A[r].Wu[n])
 *              w [G][2N][K], rows 0..N-1 gate; w_scale [G][2N]
 *  w_scale  fp32 [G][rows of W[g]] (device)
 * Other arguments, scratch, checks and the result type as moe_grouped_gemm.
 * Weight-streaming shapes only (the regime whose bytes the format halves):
 * rows_max <= 64 * G, or rows_max == 1; others give MOE_ERR_UNSUPPORTED.  The
 * codes are widened to bf16 in tensor memory (exact; the NaN codes read as
 * +-480), multiplied on the tensor cores with fp32 accumulation (on the CUDA
 * cores for one-row groups), and each row's scale is applied to the finished
 * sum. */
MOE_API int moe_grouped_gemm_w8(const void* a, const void* w, const float* w_scale, const int32_t* group_offsets,
                                int G, int rows_max, int N, int K, int act, void* out, void* ws, size_t ws_bytes,
                                cudaStream_t stream);

/* Combine: out[t] = bf16( sum_j topk_w[t,j] * y[inv_perm[t*k+j]] + shared[t] ),
 * accumulated in fp32 in slot order j = 0..k-1, then the shared row.
 *  y bf16 [T*k][H];  inv_perm int32 [T*k];  topk_w fp32 [T][k]
 *  shared bf16 [T][H] or NULL;  out bf16 [T][H]
 * Supported: H % 8 == 0, H <= 8192. */
MOE_API int moe_unpermute_combine(const void* y, const int32_t* inv_perm, const float* topk_w, const void* shared,
                          int T, int H, int k, void* out, cudaStream_t stream);

/* The whole layer: route -> permute -> gmm1(+SiLU*mul) -> gmm2 on `stream`;
 * the shared expert's two matmuls on `side` between ev_fork (recorded on
 * `stream`, waited by `side`) and ev_join (recorded on `side`, waited by
 * `stream` before the combine).  Exactly one fork and one join event per
 * call, except for one token (T == 1, k <= 8, H % 8 == 0, I_s % 8 == 0): then
 * the layer is three launches on `stream` alone (route; gate_up, which also
 * computes the shared expert's gate_up; down, which also computes the shared
 * expert's down, and the combine), and `side` and the events go unused; and
 * for 4 to 9 tokens with bf16 routed weights (I, H, I_s multiples of 128,
 * T*k <= 64*E): four launches on `stream` alone (route with the dispatch;
 * gate_up, led by the shared expert's gate_up; down, led by the shared
 * expert's down; combine), again without `side` or the events.
 * `side` and the events may be NULL when d->I_s == 0.  ws holds every
 * intermediate and the split-K scratch of the four matmuls; size it with
 * moe_workspace_bytes(d, T), align it to 256 bytes and zero-fill it before its
 * first use (calls leave the scratch counters zero).  The counters sit at the
 * same offsets for every T, so calls with different T may use one workspace
 * sized for the largest.  Calls that share a workspace must not overlap on
 * the GPU.
 *  x bf16 [T][H] (device);  out bf16 [T][H] (device) */
MOE_API size_t moe_workspace_bytes(const moe_dims* d, int T);
MOE_API int moe_forward(const moe_dims* d, const moe_weights* w, const void* x, int T, void* out, void* ws,
                size_t ws_bytes, cudaStream_t stream, cudaStream_t side, cudaEvent_t ev_fork,
                cudaEvent_t ev_join);

/* The layer with FP8 routed expert weights (see moe_grouped_gemm_w8):
 *  w_gate_up e4m3 [E][2I][H] with s_gate_up fp32 [E][2I];
 *  w_down    e4m3 [E][H][I]  with s_down    fp32 [E][H];
 * router and shared expert as in moe_weights (the shared expert stays bf16, as
 * the page on MoE multi-stream overlap runs it: bf16, unquantised). */
typedef struct {
  const float* w_router;
  const float* router_bias;
  const void* w_gate_up;
  const float* s_gate_up;
  const void* w_down;
  const float* s_down;
  const void* ws_gate_up;
  const void* ws_down;
} moe_weights_w8;

/* moe_forward with FP8 routed expert weights.  Same streams, events,
 * workspace (moe_workspace_bytes) and results as moe_forward, the routed
 * matmuls reading 1-byte weights.  Decode-sized batches: T*k <= 64*E (the
 * weights-on-M form); larger batches give MOE_ERR_UNSUPPORTED. */
MOE_API int moe_forward_w8(const moe_dims* d, const moe_weights_w8* w, const void* x, int T, void* out, void* ws,
                           size_t ws_bytes, cudaStream_t stream, cudaStream_t side, cudaEvent_t ev_fork,
                           cudaEvent_t ev_join);

/* Reads and clears the current device's status word (first device-side error
 * since the last read, MOE_OK if none).  Synchronises `stream`. */
MOE_API int moe_last_device_error(cudaStream_t stream);

/* Number of kernels the last successful call of each entry point launched on
 * the current host thread (for accounting in benchmarks). */
MOE_API int moe_last_launch_count(void);

/* Where moe_forward keeps the routing and the dispatch of a batch inside its
 * workspace: byte offsets from the start of ws, for a layer of sizes d and a
 * batch of T tokens.  After a moe_forward call on that workspace has
 * completed, the regions hold that call's
 *   topk_ids int32 [T][k], topk_w fp32 [T][k] (as moe_route returns them),
 *   expert_offsets int32 [E+1], sorted_token int32 [T*k], inv_perm int32 [T*k]
 *   (as moe_permute returns them),
 * so that a caller can inspect the layer's own expert choice and dispatch.
 * Returns MOE_ERR_INVALID / MOE_ERR_UNSUPPORTED as moe_workspace_bytes
 * refuses the sizes. */
typedef struct {
  size_t topk_ids, topk_w, expert_offsets, sorted_token, inv_perm;
} moe_workspace_offsets;
MOE_API int moe_workspace_layout(const moe_dims* d, int T, moe_workspace_offsets* out);

/* Limit, in nanoseconds, of the device-side bounded waits of kernels launched
 * from now on by any host thread (default 2e9; waits that drain copies
 * already in flight keep the default).  A wait that reaches it records
 * MOE_ERR_TIMEOUT, the kernel abandons its work and exits.  0 makes every
 * wait that is not already complete at its first test expire at once: for
 * tests of the timeout path only (outputs are then not written).  Launches
 * captured in a CUDA graph keep the limit of the capture. */
MOE_API int moe_debug_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FFN_H_ */
