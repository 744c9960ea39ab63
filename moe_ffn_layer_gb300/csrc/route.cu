// Router of the MoE FFN layer: fp32 logits l[t,e] = x[t] . Wr[e] + b[e], the k
// largest logits per token (ties to the lower expert id), reported in
// ascending id order, and weights = softmax over the k chosen logits (equal to
// the softmax over all E experts renormalised over the chosen k).
//
// The layer's routed experts are chosen per token before dispatch ("Ascend
// 910C LLM inference optimisation, part 2" (Dewu Tech), section on MoE
// multi-stream overlap: dispatch -> gmm1 -> gmm2 -> combine); the router's
// precision (fp32), the top-k and the renormalisation are the layer's
// definition in its benchmark shapes.
//
// Logit kernels:
//   T <= 16   router_gemv: one warp per (expert, quarter of H), every token at
//             once; streams Wr (E*H*4 bytes) once.  Decode shapes.
//   T >  16   router_tile: fp32 SIMT tile GEMM, 64 tokens x 64 experts per CTA.
// Then topk_softmax: one warp per token.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kGemvMaxT = 16;
constexpr int kGemvSlices = 4;   // warps sharing one expert's dot products
constexpr int kGemvExpertsPerCta = 2;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// grid: ceil(E / kGemvExpertsPerCta) CTAs of kGemvExpertsPerCta * kGemvSlices warps.
// Warp (e, s) sums h in {s*256 + lane*8 + i*kGemvSlices*256 .. +8}; the slices are
// added in slice order, so the result does not depend on scheduling.
__global__ void __launch_bounds__(kGemvExpertsPerCta* kGemvSlices * 32)
    router_gemv_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ wr,
                       const float* __restrict__ bias, int T, int H, int E, float* __restrict__ logits) {
  __shared__ float part[kGemvExpertsPerCta][kGemvSlices][kGemvMaxT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int le = warp / kGemvSlices, s = warp % kGemvSlices;
  const int e = blockIdx.x * kGemvExpertsPerCta + le;
  float acc[kGemvMaxT];
#pragma unroll
  for (int t = 0; t < kGemvMaxT; ++t) acc[t] = 0.f;
  if (e < E) {
    const float* w = wr + static_cast<size_t>(e) * H;
#pragma unroll 2
    for (int h0 = s * 256 + lane * 8; h0 < H; h0 += kGemvSlices * 256) {
      const float4 w0 = __ldg(reinterpret_cast<const float4*>(w + h0));
      const float4 w1 = __ldg(reinterpret_cast<const float4*>(w + h0 + 4));
#pragma unroll
      for (int t = 0; t < kGemvMaxT; ++t) {
        if (t < T) {
          const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H + h0));
          float f[8];
          bf16x8_to_f32(xv, f);
          float a = acc[t];
          a = fmaf(f[0], w0.x, a); a = fmaf(f[1], w0.y, a); a = fmaf(f[2], w0.z, a); a = fmaf(f[3], w0.w, a);
          a = fmaf(f[4], w1.x, a); a = fmaf(f[5], w1.y, a); a = fmaf(f[6], w1.z, a); a = fmaf(f[7], w1.w, a);
          acc[t] = a;
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kGemvMaxT; ++t) {
    float v = acc[t];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) part[le][s][t] = v;
  }
  __syncthreads();
  if (e < E && s == 0 && lane < T) {
    float v = 0.f;
#pragma unroll
    for (int q = 0; q < kGemvSlices; ++q) v += part[le][q][lane];
    if (bias) v += bias[e];
    logits[static_cast<size_t>(lane) * E + e] = v;
  }
}

// fp32 SIMT GEMM: logits[T][E] = x[T][H] . Wr[E][H]^T (+ b).  CTA tile 64 x 64,
// K chunk 32, 256 threads each owning a 4 x 4 block of outputs.
constexpr int kRT = 64, kRE = 64, kRK = 32;

__global__ void __launch_bounds__(256)
    router_tile_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ wr,
                       const float* __restrict__ bias, int T, int H, int E, float* __restrict__ logits) {
  __shared__ float xs[kRK][kRT + 4];
  __shared__ float ws[kRK][kRE + 4];
  const int t0 = blockIdx.x * kRT, e0 = blockIdx.y * kRE;
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;   // 16 x 16 threads
  float acc[4][4] = {};
  for (int k0 = 0; k0 < H; k0 += kRK) {
    {  // x tile: 64 rows x 32 bf16 = 256 x uint4 (8 bf16 each)
      const int r = tid >> 2, c = (tid & 3) * 8;
      float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (t0 + r < T && k0 + c < H) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t0 + r) * H + k0 + c));
        bf16x8_to_f32(v, f);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[c + i][r] = f[i];
    }
#pragma unroll
    for (int p = 0; p < 2; ++p) {  // Wr tile: 64 rows x 32 fp32 = 512 x float4
      const int idx = tid + p * 256;
      const int r = idx >> 3, c = (idx & 7) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e0 + r < E && k0 + c < H) v = __ldg(reinterpret_cast<const float4*>(wr + static_cast<size_t>(e0 + r) * H + k0 + c));
      ws[c + 0][r] = v.x; ws[c + 1][r] = v.y; ws[c + 2][r] = v.z; ws[c + 3][r] = v.w;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kRK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { a[i] = xs[kk][ty * 4 + i]; b[i] = ws[kk][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) logits[static_cast<size_t>(t) * E + e] = acc[i][j] + (bias ? bias[e] : 0.f);
    }
  }
}

// One warp per token: k rounds of a warp arg-max over the E logits (larger
// value wins, equal values go to the lower id), then the chosen ids are sorted
// ascending and w_j = exp(l_j - max) / sum_i exp(l_i - max) over the chosen k.
constexpr int kTopkMaxPerLane = kMaxExperts / 32;

__global__ void __launch_bounds__(256)
    topk_softmax_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ topk_ids,
                        float* __restrict__ topk_w) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  float v[kTopkMaxPerLane];
  const float* l = logits + static_cast<size_t>(t) * E;
#pragma unroll
  for (int i = 0; i < kTopkMaxPerLane; ++i) {
    const int e = i * 32 + lane;
    v[i] = e < E ? l[e] : -INFINITY;
  }
  uint32_t taken = 0;   // bit i: element i of this lane already chosen
  int ids[kMaxTopK];
  float vals[kMaxTopK];
#pragma unroll 1
  for (int r = 0; r < k; ++r) {
    float best = -INFINITY;
    int bid = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kTopkMaxPerLane; ++i) {
      const int e = i * 32 + lane;
      if (e < E && !(taken >> i & 1u) && (v[i] > best || (v[i] == best && e < bid))) { best = v[i]; bid = e; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bid, o);
      if (ob > best || (ob == best && oi < bid)) { best = ob; bid = oi; }
    }
    ids[r] = bid;
    vals[r] = best;
    if (bid < E && (bid & 31) == lane) taken |= 1u << (bid >> 5);
  }
  if (lane != 0) return;
  // insertion sort of the chosen (id, logit) pairs by id
  for (int i = 1; i < k; ++i) {
    const int ci = ids[i];
    const float cv = vals[i];
    int j = i - 1;
    while (j >= 0 && ids[j] > ci) { ids[j + 1] = ids[j]; vals[j + 1] = vals[j]; --j; }
    ids[j + 1] = ci;
    vals[j + 1] = cv;
  }
  float m = -INFINITY;
  for (int i = 0; i < k; ++i) m = fmaxf(m, vals[i]);
  float p[kMaxTopK];
  float s = 0.f;
  for (int i = 0; i < k; ++i) { p[i] = expf(vals[i] - m); s += p[i]; }
  const float inv = 1.0f / s;
  for (int i = 0; i < k; ++i) {
    topk_ids[static_cast<size_t>(t) * k + i] = ids[i];
    topk_w[static_cast<size_t>(t) * k + i] = p[i] * inv;
  }
}

}  // namespace

size_t route_ws_bytes(int T, int E) { return align_up(static_cast<size_t>(T) * E * sizeof(float)); }

int route_launch(const void* x, const float* w_router, const float* bias, int T, int H, int E, int k,
                 int32_t* topk_ids, float* topk_w, float* logits_ws, cudaStream_t stream, int* launches) {
  if (T == 0) return MOE_OK;
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  if (T <= kGemvMaxT) {
    const int grid = (E + kGemvExpertsPerCta - 1) / kGemvExpertsPerCta;
    router_gemv_kernel<<<grid, kGemvExpertsPerCta * kGemvSlices * 32, 0, stream>>>(xb, w_router, bias, T, H, E,
                                                                                   logits_ws);
  } else {
    dim3 grid((T + kRT - 1) / kRT, (E + kRE - 1) / kRE);
    router_tile_kernel<<<grid, 256, 0, stream>>>(xb, w_router, bias, T, H, E, logits_ws);
  }
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  ++*launches;
  topk_softmax_kernel<<<(T + 7) / 8, 256, 0, stream>>>(logits_ws, T, E, k, topk_ids, topk_w);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  ++*launches;
  return MOE_OK;
}

}  // namespace moe
