// C ABI of the MoE FFN layer forward: argument checks, workspace layout and
// the two-stream orchestration of moe_forward.
//
// Orchestration ("Ascend 910C LLM inference optimisation, part 2" (Dewu Tech),
// section on MoE multi-stream overlap): the shared expert reads the same
// hidden states as the routed experts and nothing of theirs, so its gate_up
// and down matmuls run on a side stream, forked from the main stream by one
// event and joined back by one event just before the combine.  The same page
// drops the per-step dispatch/combine/gmm2 events once the overlap exists and
// preallocates events instead of creating them per step: here the caller owns
// exactly two events and the library creates none.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

__device__ int g_status;   // first device-side error since the last read, per device

thread_local int t_last_launches = 0;

// Where a batch of more than 16 tokens forks the shared expert: 0 before the
// router, 1 after the router, 2 after the dispatch.  Both the shared matmuls
// and the router's tensor-core logits want every SM; forking after the router
// lets the shared matmuls overlap the top-k, the dispatch and the row copy,
// which leave the tensor cores idle (measured: prefill T=8192 850 -> 822 us,
// batched decode T=256 187 -> 180 us).  A large router (T*E*H >= 2^33, e.g.
// T=16384, E=256, H=4096) leaves enough idle SMs of its own that forking
// before it is better (4507 -> 4403 us there; the T=8192, E=128 prefill loses
// 759 -> 791 us).
// Batches whose shared expert runs as the leading phase of the routed matmul
// launches (see forward_impl).
constexpr int kLeadMinT = 4;
constexpr int kLeadMaxT = 9;

int fork_stage(const moe_dims* d, int T) {
  return static_cast<double>(T) * d->E * d->H >= 8589934592.0 ? 0 : 1;
}

std::atomic<uint64_t> g_wait_limit_ns{moe::kWaitTimeoutNs};

struct DevInfo {
  int* status = nullptr;
  int sms = 0;
  void* ctx = nullptr;   // the context the status address belongs to
  bool init = false;
};
constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
std::mutex g_mu;

int dev_info(DevInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  void* ctx = nullptr;
  if (moe::current_context(&ctx) != MOE_OK) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& d = g_dev[dev];
  // the status word's address is looked up once per context (a device reset
  // makes a new context, which holds its own copy of the word)
  if (!d.init || d.ctx != ctx || !ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (!ctx && moe::current_context(&ctx) != MOE_OK) return MOE_ERR_CUDA;   // set up by the lookup
    d.status = static_cast<int*>(p);
    d.ctx = ctx;
    d.init = true;
  }
  *out = &d;
  return MOE_OK;
}

constexpr size_t kRouteTicketBytes = 256;   // moe_route's ws: [ticket | logits scratch]

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Every intermediate of moe_forward, 256-byte aligned, in one caller-owned buffer.
struct Layout {
  size_t ctr_main, ctr_side, route_ticket;   // counters: first, at offsets that do not depend on T
  size_t gemm_main, gemm_main_bytes, gemm_side, gemm_side_bytes;
  size_t logits, ids, w, offsets, sorted, inv, pcounts, xperm, h, y, hs, s, total;
};

Layout layout(const moe_dims* d, int T) {
  Layout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t r = o;
    o += moe::align_up(bytes);
    return r;
  };
  const size_t Tk = static_cast<size_t>(T) * d->k;
  // split-K scratch: one set for the routed pair (main stream), one for the
  // shared pair (side stream), so the two streams never share counters.  The
  // counters come first, at the same offsets for every T, so that calls with
  // different T can share one workspace in turn: the region that holds one
  // call's counters never holds another call's data.
  const int rows = T * d->k;
  L.gemm_main_bytes = std::max(moe::grouped_gemm_partial_bytes(d->E, rows, d->I, 1),
                               moe::grouped_gemm_partial_bytes(d->E, rows, d->H, 0));
  L.gemm_side_bytes = d->I_s ? std::max(moe::grouped_gemm_partial_bytes(1, T, d->I_s, 1),
                                        moe::grouped_gemm_partial_bytes(1, T, d->H, 0))
                             : 0;
  L.ctr_main = take(moe::grouped_gemm_counter_region_bytes());
  L.ctr_side = take(moe::grouped_gemm_counter_region_bytes());
  L.route_ticket = take(sizeof(unsigned int));
  L.gemm_main = take(L.gemm_main_bytes);
  L.gemm_side = take(L.gemm_side_bytes);
  L.logits = take(moe::route_ws_bytes(T, d->H, d->E));
  L.ids = take(Tk * 4);
  L.w = take(Tk * 4);
  L.offsets = take((static_cast<size_t>(d->E) + 1) * 4);
  L.sorted = take(Tk * 4);
  L.inv = take(Tk * 4);
  L.pcounts = take(moe::permute_ws_bytes(T, d->E));
  // decode sizes gather the dispatched rows inside gmm1; larger batches copy them
  L.xperm = take(T <= moe::route_small_max_tokens() ? 0 : Tk * d->H * 2);
  L.h = take(Tk * d->I * 2);
  L.y = take(Tk * d->H * 2);
  L.hs = take(static_cast<size_t>(T) * d->I_s * 2);
  L.s = take(static_cast<size_t>(T) * d->H * 2);
  L.total = o;
  return L;
}

int check_dims(const moe_dims* d) {
  if (!d) return MOE_ERR_INVALID;
  if (d->H <= 0 || d->E <= 0 || d->k <= 0 || d->I <= 0 || d->I_s < 0) return MOE_ERR_INVALID;
  if (d->k > d->E) return MOE_ERR_INVALID;
  if (d->E > moe::kMaxExperts || d->k > moe::kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (d->H % 64 || d->I % 64 || d->I_s % 64) return MOE_ERR_UNSUPPORTED;
  if (d->E > moe::grouped_gemm_max_groups()) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace

namespace moe {

void set_last_launches(int n) { t_last_launches = n; }

int current_context(void** ctx) {
  using GetCtxFn = CUresult (*)(CUcontext*);
  static GetCtxFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<GetCtxFn>(p);
  });
  if (!fn) return MOE_ERR_CUDA;
  CUcontext c = nullptr;   // null until the runtime has set up the device
  if (fn(&c) != CUDA_SUCCESS) return MOE_ERR_CUDA;
  *ctx = c;
  return MOE_OK;
}

bool device_local(const void* p) {
  if (!p) return false;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();   // a pointer the runtime does not know: clear the error the query left
    return false;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  return a.type == cudaMemoryTypeDevice && a.device == dev;
}

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

int current_device_info(int** status, int* num_sms) {
  DevInfo* di = nullptr;
  const int rc = dev_info(&di);
  if (rc) return rc;
  *status = di->status;
  *num_sms = di->sms;
  return MOE_OK;
}
}  // namespace moe

extern "C" {

size_t moe_route_workspace_bytes(int T, int H, int E) {
  if (T < 0 || H <= 0 || E <= 0) return 0;
  return kRouteTicketBytes + moe::route_ws_bytes(T, H, E);
}

int moe_route(const void* x, const float* w_router, const float* bias, int T, int H, int E, int k,
              int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes, cudaStream_t stream) {
  t_last_launches = 0;
  if (T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_INVALID;
  if (E > moe::kMaxExperts || k > moe::kMaxTopK || H % 8) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !topk_ids || !topk_w || !ws) return MOE_ERR_INVALID;
  if (!al16(x) || !al16(w_router) || !al16(ws) || (reinterpret_cast<uintptr_t>(topk_ids) & 3u) ||
      (reinterpret_cast<uintptr_t>(topk_w) & 3u) || (reinterpret_cast<uintptr_t>(bias) & 3u))
    return MOE_ERR_UNSUPPORTED;
  if (ws_bytes < kRouteTicketBytes + moe::route_ws_bytes(T, H, E)) return MOE_ERR_WORKSPACE;
  DevInfo* di = nullptr;
  int rc = dev_info(&di);
  if (rc) return rc;
  int n = 0;
  // ws = [ticket counter | logits scratch]; the counter is cleared here, so ws
  // may hold anything on entry
  unsigned int* ticket = static_cast<unsigned int*>(ws);
  if (T <= moe::route_small_max_tokens() && cudaMemsetAsync(ticket, 0, sizeof(unsigned int), stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  rc = moe::route_launch(x, w_router, bias, T, H, E, k, topk_ids, topk_w,
                         reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kRouteTicketBytes), ticket, nullptr,
                         di->status, di->sms, stream, &n);
  t_last_launches = n;
  return rc;
}

size_t moe_permute_workspace_bytes(int T, int E) {
  if (T < 0 || E <= 0) return 0;
  return moe::permute_ws_bytes(T, E);
}

int moe_permute(const int32_t* topk_ids, const void* x, int T, int H, int E, int k, int32_t* expert_offsets,
                int32_t* sorted_token, int32_t* inv_perm, void* x_perm, void* ws, size_t ws_bytes,
                cudaStream_t stream) {
  t_last_launches = 0;
  if (T < 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_INVALID;
  if (E > moe::kMaxExperts || static_cast<long long>(T) * k > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
  if (x_perm && (H <= 0)) return MOE_ERR_INVALID;
  if (x_perm && H % 8) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!topk_ids || !expert_offsets || !sorted_token || !inv_perm) return MOE_ERR_INVALID;
  if (x_perm && (!x || !al16(x) || !al16(x_perm))) return x ? MOE_ERR_UNSUPPORTED : MOE_ERR_INVALID;
  const size_t need = moe::permute_ws_bytes(T, E);
  if (need && (!ws || ws_bytes < need)) return MOE_ERR_WORKSPACE;
  DevInfo* di = nullptr;
  int rc = dev_info(&di);
  if (rc) return rc;
  int n = 0;
  rc = moe::permute_launch(topk_ids, x, T, H, E, k, expert_offsets, sorted_token, inv_perm, x_perm,
                           static_cast<int32_t*>(ws), di->status, di->sms, stream, &n);
  t_last_launches = n;
  return rc;
}

size_t moe_grouped_gemm_workspace_bytes(int G, int rows_max, int N, int K, int act) {
  if (G <= 0 || rows_max < 0 || N <= 0 || K <= 0 || (act != 0 && act != 1)) return 0;
  return moe::grouped_gemm_ws_bytes(G, rows_max, N, act);
}

int moe_grouped_gemm(const void* a, const void* w, const int32_t* group_offsets, int G, int rows_max, int N, int K,
                     int act, void* out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  t_last_launches = 0;
  if (G <= 0 || rows_max < 0 || N <= 0 || K <= 0 || (act != 0 && act != 1)) return MOE_ERR_INVALID;
  if (!group_offsets && G != 1) return MOE_ERR_INVALID;
  if (G > moe::grouped_gemm_max_groups() || N % 64 || K % 64) return MOE_ERR_UNSUPPORTED;
  if (rows_max == 0) return MOE_OK;
  if (!a || !w || !out) return MOE_ERR_INVALID;
  if (!al16(a) || !al16(w) || !al16(out) || (reinterpret_cast<uintptr_t>(group_offsets) & 3u) ||
      (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOE_ERR_UNSUPPORTED;
  // TMA reads the operands: device memory of the current GPU only
  if (!moe::device_local(a) || !moe::device_local(w) || !moe::device_local(out)) return MOE_ERR_UNSUPPORTED;
  DevInfo* di = nullptr;
  int rc = dev_info(&di);
  if (rc) return rc;
  if (ws && ws_bytes < moe::grouped_gemm_ws_bytes(G, rows_max, N, act)) return MOE_ERR_WORKSPACE;
  int n = 0;
  const moe::GemmScratch scratch = moe::grouped_gemm_scratch(ws, ws_bytes);
  rc = moe::grouped_gemm_launch(a, w, group_offsets, G, rows_max, N, K, act, out, di->status, &scratch, di->sms,
                                stream, &n);
  t_last_launches = n;
  return rc;
}

int moe_grouped_gemm_w8(const void* a, const void* w, const float* w_scale, const int32_t* group_offsets, int G,
                        int rows_max, int N, int K, int act, void* out, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
  t_last_launches = 0;
  if (G <= 0 || rows_max < 0 || N <= 0 || K <= 0 || (act != 0 && act != 1)) return MOE_ERR_INVALID;
  if (!group_offsets && G != 1) return MOE_ERR_INVALID;
  if (G > moe::grouped_gemm_max_groups() || N % 64 || K % 64) return MOE_ERR_UNSUPPORTED;
  // 8-bit weights: groups of few rows (the weights-on-M form), decode-sized batches
  if (!moe::grouped_gemm_weights_on_m(G, rows_max, N) && rows_max != 1) return MOE_ERR_UNSUPPORTED;
  if (rows_max == 0) return MOE_OK;
  if (!a || !w || !w_scale || !out) return MOE_ERR_INVALID;
  if (!al16(a) || !al16(w) || !al16(out) || (reinterpret_cast<uintptr_t>(group_offsets) & 3u) ||
      (reinterpret_cast<uintptr_t>(w_scale) & 3u) || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOE_ERR_UNSUPPORTED;
  if (!moe::device_local(a) || !moe::device_local(w) || !moe::device_local(out)) return MOE_ERR_UNSUPPORTED;
  DevInfo* di = nullptr;
  int rc = dev_info(&di);
  if (rc) return rc;
  if (ws && ws_bytes < moe::grouped_gemm_ws_bytes(G, rows_max, N, act)) return MOE_ERR_WORKSPACE;
  int n = 0;
  const moe::GemmScratch scratch = moe::grouped_gemm_scratch(ws, ws_bytes);
  rc = moe::grouped_gemm_launch(a, w, group_offsets, G, rows_max, N, K, act, out, di->status, &scratch, di->sms,
                                stream, &n, nullptr, 0, 0, 0, w_scale);
  t_last_launches = n;
  return rc;
}

int moe_unpermute_combine(const void* y, const int32_t* inv_perm, const float* topk_w, const void* shared, int T,
                          int H, int k, void* out, cudaStream_t stream) {
  t_last_launches = 0;
  if (T < 0 || H <= 0 || k <= 0) return MOE_ERR_INVALID;
  if (k > moe::kMaxTopK || H % 8) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!y || !inv_perm || !topk_w || !out) return MOE_ERR_INVALID;
  if (!al16(y) || !al16(out) || (shared && !al16(shared))) return MOE_ERR_UNSUPPORTED;
  int n = 0;
  const int rc = moe::combine_launch(y, inv_perm, topk_w, shared, T, H, k, static_cast<long long>(T) * k, out,
                                     stream, &n);
  t_last_launches = n;
  return rc;
}

size_t moe_workspace_bytes(const moe_dims* d, int T) {
  if (check_dims(d) != MOE_OK || T < 0) return 0;
  return layout(d, T).total;
}

}  // extern "C"

namespace {

// The weights of a layer forward: routed experts in bf16 (scales null) or
// e4m3 with one fp32 scale per weight row; router and shared expert as in
// moe_weights.
struct LayerWeights {
  const float* w_router;
  const float* router_bias;
  const void* w_gate_up;
  const float* s_gate_up;
  const void* w_down;
  const float* s_down;
  const void* ws_gate_up;
  const void* ws_down;
};

int forward_impl(const moe_dims* d, const LayerWeights* w, const void* x, int T, void* out, void* ws, size_t ws_bytes,
                 cudaStream_t stream, cudaStream_t side, cudaEvent_t ev_fork, cudaEvent_t ev_join) {
  t_last_launches = 0;
  int rc = check_dims(d);
  if (rc) return rc;
  if (!w || T < 0) return MOE_ERR_INVALID;
  if (static_cast<long long>(T) * d->k > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
  const bool w8 = w->s_gate_up != nullptr;
  if (w8 && !w->s_down) return MOE_ERR_INVALID;
  // 8-bit routed weights: the weights-on-M matmuls (and one-row groups) only
  if (w8 && !moe::grouped_gemm_weights_on_m(d->E, T * d->k, d->I)) return MOE_ERR_UNSUPPORTED;
  if (w8 && !moe::grouped_gemm_weights_on_m(d->E, T * d->k, d->H)) return MOE_ERR_UNSUPPORTED;
  if (w8 && ((reinterpret_cast<uintptr_t>(w->s_gate_up) & 3u) || (reinterpret_cast<uintptr_t>(w->s_down) & 3u)))
    return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  const bool has_shared = d->I_s > 0;
  if (!x || !out || !ws || !w->w_router || !w->w_gate_up || !w->w_down) return MOE_ERR_INVALID;
  if (has_shared && (!w->ws_gate_up || !w->ws_down || !side || !ev_fork || !ev_join)) return MOE_ERR_INVALID;
  if (!al16(x) || !al16(out) || !al16(ws) || !al16(w->w_router) || !al16(w->w_gate_up) || !al16(w->w_down) ||
      (reinterpret_cast<uintptr_t>(w->router_bias) & 3u) ||
      (has_shared && (!al16(w->ws_gate_up) || !al16(w->ws_down))))
    return MOE_ERR_UNSUPPORTED;
  const Layout L = layout(d, T);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  // the matmuls read x, the weights and the workspace by TMA: device memory of the current GPU only
  if (!moe::device_local(x) || !moe::device_local(out) || !moe::device_local(ws) ||
      !moe::device_local(w->w_gate_up) || !moe::device_local(w->w_down) ||
      (has_shared && (!moe::device_local(w->ws_gate_up) || !moe::device_local(w->ws_down))))
    return MOE_ERR_UNSUPPORTED;
  DevInfo* di = nullptr;
  rc = dev_info(&di);
  if (rc) return rc;

  uint8_t* base = static_cast<uint8_t*>(ws);
  float* logits = reinterpret_cast<float*>(base + L.logits);
  int32_t* ids = reinterpret_cast<int32_t*>(base + L.ids);
  float* tw = reinterpret_cast<float*>(base + L.w);
  int32_t* offsets = reinterpret_cast<int32_t*>(base + L.offsets);
  int32_t* sorted = reinterpret_cast<int32_t*>(base + L.sorted);
  int32_t* inv = reinterpret_cast<int32_t*>(base + L.inv);
  int32_t* pcounts = reinterpret_cast<int32_t*>(base + L.pcounts);
  void* h = base + L.h;
  void* y = base + L.y;
  void* hs = base + L.hs;
  void* s = base + L.s;
  void* xperm = base + L.xperm;
  const moe::GemmScratch gmain{reinterpret_cast<int*>(base + L.ctr_main), base + L.gemm_main, L.gemm_main_bytes};
  const moe::GemmScratch gside{reinterpret_cast<int*>(base + L.ctr_side), base + L.gemm_side, L.gemm_side_bytes};
  const int rows = T * d->k;
  int n = 0;

  // One token with a shared expert: three launches and no side stream.  The
  // router lets the gate_up weight stream start at once; that launch first
  // computes the shared expert's gate_up (it needs only x) while the router
  // runs, then the routed rows; the down launch computes the shared expert's
  // down beside the routed ones and adds it in the combine.
  const bool one_token_fused = T == 1 && has_shared && d->I_s % 8 == 0 &&
                               moe::down_combine_gemv_applies(d->E, d->H, d->I, d->k) &&
                               moe::grouped_gemv_applies(d->E, d->I, d->H, 1, 1);
  // 4 to 9 tokens with a shared expert (bf16 weights): no side stream either.
  // The routed matmul launches carry the shared expert as a leading phase:
  // its gate_up streams the shared weights while the router runs (before that
  // launch's wait on the router), its down leads the routed down launch, and
  // the combine adds its row.  Every SM serves both.  Measured against the
  // side stream (decode sizes, one GPU, back to back): 2.3 us faster on
  // average over T = 4..9 (T = 8: 111.7 -> 109.2 us), slower at T = 2, 3 and
  // from 12 on, where the routing window is too short to hide the shared
  // gate_up or the larger router leaves no room beside it on its SMs.
  const bool lead_shared = !one_token_fused && T >= kLeadMinT && T <= kLeadMaxT && has_shared &&
                           !w->s_gate_up && L.gemm_side_bytes > 0 &&
                           moe::lead_phase_applies(T, d->I_s, d->H) && moe::lead_phase_applies(T, d->H, d->I_s) &&
                           moe::grouped_gemm_weights_on_m(d->E, rows, d->I) &&
                           moe::grouped_gemm_weights_on_m(d->E, rows, d->H);
  // SMs for the two streams.  At decode sizes both are weight streams that
  // run side by side for the whole call: the shared expert gets the SMs in
  // proportion to its share of the weight bytes (at least 8, at most half),
  // the routed matmuls the rest.  Larger batches give both streams every SM.
  int side_sms = di->sms, main_sms = di->sms;
  if (T <= moe::route_small_max_tokens() && has_shared && !one_token_fused && !lead_shared) {
    const double shared_bytes = 3.0 * d->I_s * d->H * 2;
    const double routed_bytes = 3.0 * d->I * d->H * 2 * std::min<long long>(d->E, static_cast<long long>(T) * d->k);
    int c = static_cast<int>(di->sms * shared_bytes / (shared_bytes + routed_bytes) + 0.5);
    c = std::max(8, std::min(c, di->sms / 2));
    side_sms = c;
    main_sms = di->sms - c;
  }
  // shared expert on the side stream, forked from `stream`
  auto fork_shared = [&]() -> int {
    if (!has_shared) return MOE_OK;
    if (cudaEventRecord(ev_fork, stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamWaitEvent(side, ev_fork, 0) != cudaSuccess) return MOE_ERR_CUDA;
    // (a token adds at most one row to a group: no group holds more than T rows)
    int r = moe::grouped_gemm_launch(x, w->ws_gate_up, nullptr, 1, T, d->I_s, d->H, 1, hs, di->status, &gside,
                                     side_sms, side, &n, nullptr, 0, 0, T);
    if (!r)
      r = moe::grouped_gemm_launch(hs, w->ws_down, nullptr, 1, T, d->H, d->I_s, 0, s, di->status, &gside,
                                   side_sms, side, &n, nullptr, 0, 0, T);
    if (r) return r;
    return cudaEventRecord(ev_join, side) != cudaSuccess ? MOE_ERR_CUDA : MOE_OK;
  };
  // routed path on `stream`: route -> dispatch -> gmm1 (+SiLU*mul) -> gmm2
  if (T <= moe::route_small_max_tokens()) {
    // decode sizes: the shared expert streams its weights while one router
    // launch routes and dispatches
    if (!one_token_fused && !lead_shared) rc = fork_shared();
    // router, top-k and counting sort in one launch
    const moe::DispatchOut dout{offsets, sorted, inv};
    if (!rc)
      rc = moe::route_launch(x, w->w_router, w->router_bias, T, d->H, d->E, d->k, ids, tw, logits,
                             reinterpret_cast<unsigned int*>(base + L.route_ticket), &dout, di->status, di->sms,
                             stream, &n, one_token_fused || lead_shared);
  } else {
    const int fork_at = fork_stage(d, T);
    if (fork_at == 0) rc = fork_shared();
    if (!rc)
      rc = moe::route_launch(x, w->w_router, w->router_bias, T, d->H, d->E, d->k, ids, tw, logits, nullptr,
                             nullptr, di->status, di->sms, stream, &n);
    if (!rc && fork_at == 1) rc = fork_shared();
    if (!rc)
      rc = moe::permute_launch(ids, x, T, d->H, d->E, d->k, offsets, sorted, inv, xperm, pcounts, di->status,
                               di->sms, stream, &n);
    if (!rc && fork_at == 2) rc = fork_shared();
  }
  const moe::LeadPhase lead_gu{x, w->ws_gate_up, T, d->I_s, d->H, hs, true, gside};
  const moe::LeadPhase lead_dn{hs, w->ws_down, T, d->H, d->I_s, s, false, gside};
  if (!rc)
    // decode sizes: gmm1 reads the dispatched rows straight from x through
    // sorted_token (TMA gather4, a few rows per stage); larger batches read the
    // permuted copy, since one producer thread issuing a gather per 4 rows
    // cannot feed full 128-row tiles
    rc = one_token_fused
             ? moe::grouped_gemv_launch(x, w->w_gate_up, w->s_gate_up, offsets, d->E, rows, d->I, d->H, 1, h,
                                        di->status, stream, &n, sorted, T, 1, di->sms, x, w->ws_gate_up, d->I_s, hs)
         : T <= moe::route_small_max_tokens()
             ? moe::grouped_gemm_launch(x, w->w_gate_up, offsets, d->E, rows, d->I, d->H, 1, h, di->status, &gmain,
                                        main_sms, stream, &n, sorted, T, 0, T, w->s_gate_up,
                                        lead_shared ? &lead_gu : nullptr)
             : moe::grouped_gemm_launch(xperm, w->w_gate_up, offsets, d->E, rows, d->I, d->H, 1, h, di->status,
                                        &gmain, di->sms, stream, &n, nullptr, 0, 0, 0, w->s_gate_up);
  // one token: gmm2 and the combine in one launch, after the join (the shared
  // expert has long finished by then: it streamed its weights during routing)
  const bool fused_tail = T == 1 && moe::down_combine_gemv_applies(d->E, d->H, d->I, d->k);
  if (!rc && !fused_tail)
    rc = moe::grouped_gemm_launch(h, w->w_down, offsets, d->E, rows, d->H, d->I, 0, y, di->status, &gmain,
                                  main_sms, stream, &n, nullptr, 0, 0, T, w->s_down, lead_shared ? &lead_dn : nullptr);
  if (rc) return rc;
  // join, then combine
  if (has_shared && !one_token_fused && !lead_shared && cudaStreamWaitEvent(stream, ev_join, 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  rc = fused_tail ? moe::down_combine_gemv_launch(h, w->w_down, w->s_down, offsets, d->E, d->H, d->I, d->k, inv, tw,
                                                  has_shared && !one_token_fused ? s : nullptr, out, di->status,
                                                  stream, &n, one_token_fused ? w->ws_down : nullptr,
                                                  one_token_fused ? hs : nullptr, d->I_s)
                  : moe::combine_launch(y, inv, tw, has_shared ? s : nullptr, T, d->H, d->k, rows, out, stream, &n);
  t_last_launches = n;
  return rc;
}

}  // namespace

extern "C" {

int moe_forward(const moe_dims* d, const moe_weights* w, const void* x, int T, void* out, void* ws,
                size_t ws_bytes, cudaStream_t stream, cudaStream_t side, cudaEvent_t ev_fork, cudaEvent_t ev_join) {
  if (!w) {
    t_last_launches = 0;
    return MOE_ERR_INVALID;
  }
  const LayerWeights lw{w->w_router, w->router_bias, w->w_gate_up, nullptr, w->w_down, nullptr, w->ws_gate_up,
                        w->ws_down};
  return forward_impl(d, &lw, x, T, out, ws, ws_bytes, stream, side, ev_fork, ev_join);
}

int moe_forward_w8(const moe_dims* d, const moe_weights_w8* w, const void* x, int T, void* out, void* ws,
                   size_t ws_bytes, cudaStream_t stream, cudaStream_t side, cudaEvent_t ev_fork, cudaEvent_t ev_join) {
  if (!w || !w->s_gate_up || !w->s_down) {
    t_last_launches = 0;
    return MOE_ERR_INVALID;
  }
  const LayerWeights lw{w->w_router, w->router_bias, w->w_gate_up, w->s_gate_up, w->w_down, w->s_down,
                        w->ws_gate_up, w->ws_down};
  return forward_impl(d, &lw, x, T, out, ws, ws_bytes, stream, side, ev_fork, ev_join);
}

int moe_last_device_error(cudaStream_t stream) {
  DevInfo* di = nullptr;
  int rc = dev_info(&di);
  if (rc) return rc;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, di->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  const int zero = 0;
  if (v != 0 && cudaMemcpy(di->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return MOE_ERR_CUDA;
  return v;
}

int moe_last_launch_count(void) { return t_last_launches; }

int moe_workspace_layout(const moe_dims* d, int T, moe_workspace_offsets* out) {
  if (!out || T < 0) return MOE_ERR_INVALID;
  const int rc = check_dims(d);
  if (rc) return rc;
  const Layout L = layout(d, T);
  out->topk_ids = L.ids;
  out->topk_w = L.w;
  out->expert_offsets = L.offsets;
  out->sorted_token = L.sorted;
  out->inv_perm = L.inv;
  return MOE_OK;
}

int moe_debug_set_wait_limit_ns(uint64_t ns) {
  g_wait_limit_ns.store(ns, std::memory_order_relaxed);
  return MOE_OK;
}

}  // extern "C"
