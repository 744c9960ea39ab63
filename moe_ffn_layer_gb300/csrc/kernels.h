// Internal launch functions of the MoE FFN library (host side).  Each checks
// nothing that the C-ABI layer has already checked, returns a moe_status and
// adds the number of kernels it launched to *launches.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// Dispatch outputs the small-T router can produce in the same launch.
struct DispatchOut {
  int32_t* offsets;
  int32_t* sorted_token;
  int32_t* inv_perm;
};

size_t route_ws_bytes(int T, int H, int E);
int route_small_max_tokens();
// logits_ws: route_ws_bytes(T, H, E) bytes.  ticket: a counter that is zero on
// entry and left zero (used for T <= route_small_max_tokens(), required there).
// dispatch != nullptr requires T <= route_small_max_tokens().
// early_release (T <= 16 form): the launch lets the next kernel of the stream
// start as soon as its own wait on the previous kernel has returned.
int route_launch(const void* x, const float* w_router, const float* bias, int T, int H, int E, int k,
                 int32_t* topk_ids, float* topk_w, float* logits_ws, unsigned int* ticket, const DispatchOut* dispatch,
                 int* status, int grid_cap, cudaStream_t stream, int* launches, bool early_release = false);

size_t permute_ws_bytes(int T, int E);
int permute_launch(const int32_t* topk_ids, const void* x, int T, int H, int E, int k, int32_t* offsets,
                   int32_t* sorted_token, int32_t* inv_perm, void* x_perm, int32_t* block_counts, int* status,
                   int num_sms, cudaStream_t stream, int* launches);

bool grouped_gemm_weights_on_m(int G, int rows_max, int N);
// Split-K scratch of the weights-on-M form: ticket counters (zero between
// calls; every call leaves the ones it used zero) and partial-sum slots.
struct GemmScratch {
  int* counters;          // grouped_gemm_counter_region_bytes() bytes, or nullptr: no split
  void* partials;
  size_t partial_bytes;
};
// Size of the counter region, the same for every shape.
size_t grouped_gemm_counter_region_bytes();
// Counter bytes (from the start of the region) a launch of this shape may use.
size_t grouped_gemm_counters_used_bytes(int G, int rows_max, int N, int act);
// Partial-slot bytes a launch needs to split with at most max_slots slots (0: default cap);
// 0 when the shape never splits.
size_t grouped_gemm_partial_bytes(int G, int rows_max, int N, int act, int max_slots = 0);
// One buffer laid out as [counter region | partial slots]; 0 when the shape never splits.
size_t grouped_gemm_ws_bytes(int G, int rows_max, int N, int act, int max_slots = 0);
GemmScratch grouped_gemm_scratch(void* ws, size_t ws_bytes);
// scratch (nullable): split-K scratch.
// a_rows (nullable): token row r of the product is row a_rows[r] of `a`, a
// [a_src_rows][K] tensor (rows fetched by TMA gather4, no permuted copy).
// max_group_rows (0: unknown): a bound on any group's rows that the caller knows.
// w_scale (nullable): w holds e4m3 codes with one fp32 scale per weight row
// (weights-on-M shapes and one-row groups only; others MOE_ERR_UNSUPPORTED).
// A leading phase of a weights-on-M launch (bf16 weights): one group of
// rows <= 16 token rows a [rows][K] times weights w ([2N][K] with SiLU*mul,
// else [N][K]) into out [rows][N], with split-K scratch of its own; early:
// it runs before the launch waits on the previous kernel of the stream, so a
// and w must not come from that kernel.
struct LeadPhase {
  const void* a;
  const void* w;
  int rows, N, K;
  void* out;
  bool early;
  GemmScratch scratch;
};
// Whether a leading phase of these sizes can join a launch (rows, N and K as above).
bool lead_phase_applies(int rows, int N, int K);
int grouped_gemm_launch(const void* a, const void* w, const int32_t* offsets, int G, int rows_max, int N, int K,
                        int act, void* out, int* status, const GemmScratch* scratch, int grid_cap,
                        cudaStream_t stream, int* launches, const int32_t* a_rows = nullptr, int a_src_rows = 0,
                        int max_slots = 0, int max_group_rows = 0, const float* w_scale = nullptr,
                        const LeadPhase* lead = nullptr);
int grouped_gemm_max_groups();
// Groups of one row (max_group_rows: a bound the caller knows, e.g. T when a
// token adds at most one row per group) run on the CUDA cores: a weight stream
// where a tensor-core tile would mostly hold padding.
bool grouped_gemv_applies(int G, int N, int K, int act, int max_group_rows);
// w_scale non-null: w holds e4m3 codes with one fp32 scale per weight row.
// grid_cap: SMs the launch may fill (0: all).
// pre_w non-null: the launch first computes pre_out[1][pre_N] =
// silu(pre_a . Wg[n]) * (pre_a . Wu[n]) with pre_w = bf16 [2 pre_N][K], before
// it waits on the previous kernel of the stream; only for a launch whose
// predecessor lets dependents start once its own wait on its predecessor has
// returned (route_launch with early_release).
int grouped_gemv_launch(const void* a, const void* w, const float* w_scale, const int32_t* offsets, int G,
                        int rows_max, int N, int K, int act, void* out, int* status, cudaStream_t stream,
                        int* launches, const int32_t* a_rows, int a_src_rows, int max_group_rows, int grid_cap = 0,
                        const void* pre_a = nullptr, const void* pre_w = nullptr, int pre_N = 0,
                        void* pre_out = nullptr);
// One token: gmm2 over its k one-row groups and the combine in one launch
// (out[H] = bf16(sum_j topk_w[j] * y_j + shared)), the same bits as the one-row
// gmm2 followed by combine_launch.  h: [k][K] rows in group order; shared
// nullable.  k <= 8.  shared_w non-null (bf16 [N][K_s], K_s % 8 == 0): the
// shared expert's down matmul of shared_h [K_s] is computed in the same
// launch and added (rounded to bf16) in place of `shared`.
bool down_combine_gemv_applies(int G, int N, int K, int k);
int down_combine_gemv_launch(const void* h, const void* w_down, const float* w_scale, const int32_t* offsets, int G,
                             int N, int K, int k, const int32_t* inv_perm, const float* topk_w, const void* shared,
                             void* out, int* status, cudaStream_t stream, int* launches,
                             const void* shared_w = nullptr, const void* shared_h = nullptr, int K_s = 0);
// logits[T][E] fp32 = x[T][H] . (hi + mid + lo)^T with wr3 = bf16 [E][3H] holding
// the three bf16 terms of the fp32 router weights in K order (hi | mid | lo);
// the x tile is re-read for each of the three.  E % 64 == 0, H % 64 == 0.
int router_gemm_launch(const void* x, const void* wr3, int T, int H, int E, float* logits, int* status, int grid_cap,
                       cudaStream_t stream, int* launches);

int combine_launch(const void* y, const int32_t* inv_perm, const float* topk_w, const void* shared, int T, int H,
                   int k, long long rows_max, void* out, cudaStream_t stream, int* launches);

// Status word and SM count of the current device (first use looks them up).
int current_device_info(int** status, int* num_sms);

// What moe_last_launch_count() reports on this host thread.
void set_last_launches(int n);

// The calling thread's current CUDA context (null before the runtime has set
// up the current device).
int current_context(void** ctx);

// True when p is device memory (cudaMemoryTypeDevice) of the current device.
bool device_local(const void* p);

// Limit of the kernels' bounded waits for launches made from now on
// (kWaitTimeoutNs unless a test lowered it).
uint64_t wait_limit_ns();

}  // namespace moe
