// moe_grouped_gemm_noalloc: the grouped matmul for callers that must not
// allocate device memory.  Its split-K scratch (the per-unit ticket counters
// and the fp32 partial accumulators) lives in a fixed array of this library's
// own device memory instead of a caller-provided buffer.
//
// The array is a file-scope static __device__ object: every GPU on which the
// library's kernels are loaded holds it, MOE_NOALLOC_SCRATCH_BYTES in size,
// until the process exits.  Host code cannot use the array's name as a device
// address, so the first call on each device asks the runtime for the address
// (cudaGetSymbolAddress, with that device current) and keeps it together with
// the context it belongs to; a call made in another context (after a device
// reset, say) looks it up again.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;
constexpr int kScratchSlots = 1024;   // split-K partial slots that fit the array
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

void* g_scratch_ptr[kMaxDevices] = {};
void* g_scratch_ctx[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the array on the current device (looked up once per
// device and context).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  void* ctx = nullptr;
  if (moe::current_context(&ctx) != MOE_OK) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev] || !ctx || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    if (!ctx && moe::current_context(&ctx) != MOE_OK) return MOE_ERR_CUDA;   // set up by the lookup
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

int moe_grouped_gemm_noalloc(const void* a, const void* w, const int32_t* group_offsets, int G, int rows_max, int N,
                             int K, int act, void* out, cudaStream_t stream) {
  moe::set_last_launches(0);
  if (G <= 0 || rows_max < 0 || N <= 0 || K <= 0 || (act != 0 && act != 1)) return MOE_ERR_INVALID;
  if (!group_offsets && G != 1) return MOE_ERR_INVALID;
  if (G > moe::grouped_gemm_max_groups() || N % 64 || K % 64) return MOE_ERR_UNSUPPORTED;
  if (rows_max == 0) return MOE_OK;
  if (!a || !w || !out) return MOE_ERR_INVALID;
  if (!al16(a) || !al16(w) || !al16(out) || (reinterpret_cast<uintptr_t>(group_offsets) & 3u))
    return MOE_ERR_UNSUPPORTED;
  // TMA reads the operands: device memory of the current GPU only
  if (!moe::device_local(a) || !moe::device_local(w) || !moe::device_local(out)) return MOE_ERR_UNSUPPORTED;
  // problems whose split-K scratch does not fit the fixed array are refused
  const size_t need = moe::grouped_gemm_ws_bytes(G, rows_max, N, act, kScratchSlots);
  if (need > kScratchBytes) return MOE_ERR_WORKSPACE;
  int* status = nullptr;
  int sms = 0;
  int rc = moe::current_device_info(&status, &sms);
  if (rc) return rc;
  void* scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc) return rc;
  // the array keeps whatever the previous call left: the ticket counters this
  // launch may use must start at zero, so clear them (the partial slots are
  // always written before they are read)
  const size_t counters = moe::grouped_gemm_counters_used_bytes(G, rows_max, N, act);
  if (need && counters && cudaMemsetAsync(scratch, 0, counters, stream) != cudaSuccess) return MOE_ERR_CUDA;
  const moe::GemmScratch s = moe::grouped_gemm_scratch(scratch, kScratchBytes);
  int n = 0;
  rc = moe::grouped_gemm_launch(a, w, group_offsets, G, rows_max, N, K, act, out, status, &s, sms, stream, &n,
                                nullptr, 0, kScratchSlots);
  // launches counted as moe_grouped_gemm counts them (the counter clear is a memset, not a kernel)
  if (rc == MOE_OK) moe::set_last_launches(n);
  return rc;
}

}  // extern "C"
