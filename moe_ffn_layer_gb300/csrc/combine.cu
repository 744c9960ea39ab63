// Combine of the MoE FFN layer: out[t] = bf16( sum_j w[t,j] * y[inv_perm[t*k+j]]
// + shared[t] ), fp32 accumulation in slot order j = 0..k-1, then the shared
// expert's row, rounded once to bf16 (round to nearest even).
//
// "combine" closes the routed path (dispatch -> gmm1 -> gmm2 -> combine) and
// the shared expert's output joins it there ("Ascend 910C LLM inference
// optimisation, part 2" (Dewu Tech), section on MoE multi-stream overlap); at
// one expert-parallel rank it is a single weighted reduction per token.
//
// One CTA per token; each thread handles 8 consecutive columns per step with
// 16-byte loads of the k expert rows and 16-byte stores.  Small batches (few
// CTAs, latency-bound) issue every load of a step before the first add; large
// batches keep one load in flight per thread, which keeps registers low and
// many CTAs resident.  Both add in slot order.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kCombineThreads = 256;

constexpr int kCombineBatchedMaxT = 1024;   // tokens up to which every load of a step goes out at once

template <bool BATCHED>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ inv_perm,
                   const float* __restrict__ topk_w, const uint4* __restrict__ shared, int T, int H, int k,
                   long long rows_max, uint4* __restrict__ out) {
  __shared__ int s_row[kMaxTopK];
  __shared__ float s_w[kMaxTopK];
  chain_wait();
  const ChainReleaseAtExit release_next;
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    const int r = inv_perm[static_cast<size_t>(t) * k + threadIdx.x];
    // a pair the permute rejected (row -1) or a row out of range adds nothing
    s_row[threadIdx.x] = (r >= 0 && r < rows_max) ? r : -1;
    s_w[threadIdx.x] = topk_w[static_cast<size_t>(t) * k + threadIdx.x];
  }
  __syncthreads();
  const int vec = H / 8;
  auto add_row = [](float (&acc)[8], float w, const uint4& v) {
    acc[0] = fmaf(w, bf16_lo(v.x), acc[0]); acc[1] = fmaf(w, bf16_hi(v.x), acc[1]);
    acc[2] = fmaf(w, bf16_lo(v.y), acc[2]); acc[3] = fmaf(w, bf16_hi(v.y), acc[3]);
    acc[4] = fmaf(w, bf16_lo(v.z), acc[4]); acc[5] = fmaf(w, bf16_hi(v.z), acc[5]);
    acc[6] = fmaf(w, bf16_lo(v.w), acc[6]); acc[7] = fmaf(w, bf16_hi(v.w), acc[7]);
  };
  for (int c = threadIdx.x; c < vec; c += kCombineThreads) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    uint4 sv = make_uint4(0, 0, 0, 0);
    if (BATCHED) {
      uint4 v[kMaxTopK];
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j)
        if (j < k && s_row[j] >= 0) v[j] = __ldg(y + static_cast<size_t>(s_row[j]) * vec + c);
      if (shared) sv = __ldg(shared + static_cast<size_t>(t) * vec + c);
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j)
        if (j < k && s_row[j] >= 0) add_row(acc, s_w[j], v[j]);
    } else {
      for (int j = 0; j < k; ++j) {
        const int r = s_row[j];
        if (r < 0) continue;
        add_row(acc, s_w[j], __ldg(y + static_cast<size_t>(r) * vec + c));
      }
      if (shared) sv = __ldg(shared + static_cast<size_t>(t) * vec + c);
    }
    if (shared) {
      acc[0] += bf16_lo(sv.x); acc[1] += bf16_hi(sv.x); acc[2] += bf16_lo(sv.y); acc[3] += bf16_hi(sv.y);
      acc[4] += bf16_lo(sv.z); acc[5] += bf16_hi(sv.z); acc[6] += bf16_lo(sv.w); acc[7] += bf16_hi(sv.w);
    }
    out[static_cast<size_t>(t) * vec + c] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                                       pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
  }
}

}  // namespace

int combine_launch(const void* y, const int32_t* inv_perm, const float* topk_w, const void* shared, int T, int H,
                   int k, long long rows_max, void* out, cudaStream_t stream, int* launches) {
  if (T == 0) return MOE_OK;
  auto kernel = T <= kCombineBatchedMaxT ? combine_kernel<true> : combine_kernel<false>;
  if (launch_chained(kernel, dim3(T), dim3(kCombineThreads), 0, stream, static_cast<const uint4*>(y), inv_perm, topk_w,
                     static_cast<const uint4*>(shared), T, H, k, rows_max, static_cast<uint4*>(out)) != cudaSuccess)
    return MOE_ERR_CUDA;
  ++*launches;
  return MOE_OK;
}

}  // namespace moe
