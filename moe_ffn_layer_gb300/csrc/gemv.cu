// Grouped matmul for groups of one token row (decode at T = 1): gmm1
// (+SiLU*mul) and gmm2 of the MoE FFN layer ("Ascend 910C LLM inference
// optimisation, part 2" (Dewu Tech), section on MoE multi-stream overlap: the
// routed path is dispatch -> gmm1 -> gmm2 -> combine), computed on the CUDA
// cores instead of the tensor cores.
//
// With one token row per expert each weight element is used by one
// multiply-add: the work is a weight stream (HBM-bound), and a tensor-core MMA
// with 16 token columns would spend its issue slots on padding.  (Measured on
// GB300: faster than the tensor-core form at one row, slower at two and four,
// where the per-element unpacking and FMAs start to bind; the kernel keeps a
// row count R so that the bound stays explicit.)
// A warp owns one output column of its group (gate and up rows with SiLU*mul)
// or kRowsDown output columns (plain), reads those weight rows once with
// 16-byte loads (kSteps strides of K in flight), keeps one fp32 sum per
// (weight row, token row) per lane, and adds the lanes with a fixed butterfly:
// deterministic, fp32 accumulation.
//
// At one token the step is latency-bound, so the grid is persistent (resident
// CTAs walk the (non-empty group, output block) items) and each CTA lists the
// non-empty groups once, with all offsets loaded in one round.  For one token
// gmm2 and the combine also run as one launch (down_combine_gemv_kernel).
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kMaxGemvGroups = 1024;
constexpr int kRowsDown = 2;        // output columns per warp without SiLU*mul
constexpr int kSteps = 8;           // K strides (256 elements each) whose loads a lane issues together
constexpr int kGemvThreads = 256;

__device__ __forceinline__ void bf16x8(const uint4& v, float (&f)[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Eight consecutive weights of a row: bf16 (WT 0, 16 bytes) or e4m3 codes (WT
// 1, 8 bytes; the row's scale is applied to the finished dot product).
template <int WT>
struct WeightChunk;
template <>
struct WeightChunk<0> {
  using Vec = uint4;
  __device__ static Vec load(const uint8_t* row, int k) { return __ldg(reinterpret_cast<const uint4*>(row + 2 * k)); }
  __device__ static void to_f32(const Vec& v, float (&f)[8]) { bf16x8(v, f); }
  static constexpr int kBytes = 2;
};
template <>
struct WeightChunk<1> {
  using Vec = uint2;
  __device__ static Vec load(const uint8_t* row, int k) { return __ldg(reinterpret_cast<const uint2*>(row + k)); }
  __device__ static void to_f32(const Vec& v, float (&f)[8]) { e4m3x8_to_f32(v, f); }
  static constexpr int kBytes = 1;
};

// The non-empty groups in ascending order into s_groups, their first rows and
// row counts into s_r0 / s_nr, their number into *s_count (every thread of the
// CTA takes part; one round of offset loads).  A group with more rows than
// max_rows, or offsets out of range, is a device-side error: recorded,
// skipped.  Without offsets the one group holds rows_max rows.
__device__ __forceinline__ void list_groups(const int32_t* __restrict__ offsets, int G, int rows_max, int max_rows,
                                            int* status, int* s_groups, int* s_r0, int* s_nr, int* s_count) {
  constexpr int kChunks = kMaxGemvGroups / kGemvThreads;
  constexpr int kWarps = kGemvThreads / 32;
  static_assert(kChunks * kWarps == 32, "one warp scans the (chunk, warp) counts");
  __shared__ int s_base[kChunks * kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int lo[kChunks], hi[kChunks];
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int g = c * kGemvThreads + threadIdx.x;
    lo[c] = 0;
    hi[c] = 0;
    if (g < G) {
      lo[c] = offsets ? __ldg(offsets + g) : 0;
      hi[c] = offsets ? __ldg(offsets + g + 1) : rows_max;
    }
  }
  uint32_t mask[kChunks];
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int g = c * kGemvThreads + threadIdx.x;
    bool live = false;
    if (g < G) {
      const bool bad = lo[c] < 0 || hi[c] < lo[c] || hi[c] > rows_max || hi[c] - lo[c] > max_rows;
      if (bad) set_status(status, MOE_ERR_DEVICE_CHECK);
      live = !bad && hi[c] > lo[c];
    }
    mask[c] = __ballot_sync(0xffffffffu, live);
    if (lane == 0) s_base[c * kWarps + warp] = __popc(mask[c]);
  }
  __syncthreads();
  if (warp == 0) {   // exclusive prefix over (chunk, warp) = ascending group order
    const int v = s_base[lane];
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    s_base[lane] = incl - v;
    if (lane == 31) *s_count = incl;
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < kChunks; ++c)
    if (mask[c] >> lane & 1u) {
      const int slot = s_base[c * kWarps + warp] + __popc(mask[c] & ((1u << lane) - 1u));
      s_groups[slot] = c * kGemvThreads + threadIdx.x;
      s_r0[slot] = lo[c];
      s_nr[slot] = hi[c] - lo[c];
    }
  __syncthreads();
}

// ACT 1: out[r][n] = silu(a[r].Wg[n]) * (a[r].Wu[n]), W[g] = [2N][K] (gate rows
// first); ACT 0: out[r][n] = a[r].W[g][n], W[g] = [N][K].  Token row r of the
// product is row a_rows[r] of `a` when a_rows is given, else row r.  R >= the
// rows of any group (1, 2 or 4).  WT 1: W holds e4m3 codes and wscale one fp32
// scale per weight row ([G][2N] or [G][N]), applied to each dot product.
// One warp, one item: output block n0 (one column with SiLU*mul, kRowsDown
// without) of group g, whose token rows are r0 .. r0 + nr - 1.
// src (optional): the R source rows of `a` for the group's token rows, already
// resolved (then a_rows is not read).
template <int ACT, int R, int WT>
__device__ __forceinline__ void gemv_item(const __nv_bfloat16* __restrict__ a, const uint8_t* __restrict__ w,
                                          const float* __restrict__ wscale, int g, int n0, int r0, int nr, int N,
                                          int K, const int32_t* __restrict__ a_rows, int a_src_rows, int rows_max,
                                          __nv_bfloat16* __restrict__ out, const int* src_rows = nullptr) {
  using WC = WeightChunk<WT>;
  constexpr int NW = ACT == 1 ? 2 : kRowsDown;   // weight rows per warp
  constexpr int NPW = ACT == 1 ? 1 : kRowsDown;  // output columns per warp
  const int lane = threadIdx.x & 31;
  // this warp's weight rows and token rows (rows past nr repeat the last one)
  const size_t wrows = ACT == 1 ? 2 * static_cast<size_t>(N) : N;
  const uint8_t* wr[NW];
  size_t wrow_idx[NW];
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    wrow_idx[i] = static_cast<size_t>(g) * wrows + (ACT == 1 ? (i == 0 ? n0 : N + n0) : n0 + i);
    wr[i] = w + wrow_idx[i] * K * WC::kBytes;
  }
  const __nv_bfloat16* ar[R];
#pragma unroll
  for (int j = 0; j < R; ++j) {
    int src;
    if (src_rows) {
      src = src_rows[j];
    } else {
      const int r = r0 + (j < nr ? j : nr - 1);
      src = a_rows ? a_rows[r] : r;
      if (src < 0 || src >= (a_rows ? a_src_rows : rows_max)) src = 0;   // checked upstream; never out of range
    }
    ar[j] = a + static_cast<size_t>(src) * K;
  }
  float acc[NW][R];
#pragma unroll
  for (int i = 0; i < NW; ++i)
#pragma unroll
    for (int j = 0; j < R; ++j) acc[i][j] = 0.f;
  // kSteps strides of K per pass: every load of a pass goes out before its
  // first FMA (a lane keeps kSteps * (NW + R) 16-byte loads in flight)
  for (int kb = lane * 8; kb < K; kb += 256 * kSteps) {
    typename WC::Vec wv[kSteps][NW];
    uint4 av[kSteps][R];
#pragma unroll
    for (int u = 0; u < kSteps; ++u) {
      const int k0 = kb + u * 256;
      if (k0 < K) {
#pragma unroll
        for (int i = 0; i < NW; ++i) wv[u][i] = WC::load(wr[i], k0);
#pragma unroll
        for (int j = 0; j < R; ++j) av[u][j] = __ldg(reinterpret_cast<const uint4*>(ar[j] + k0));
      }
    }
#pragma unroll
    for (int u = 0; u < kSteps; ++u) {
      if (kb + u * 256 >= K) break;
#pragma unroll
      for (int j = 0; j < R; ++j) {
        float af[8];
        bf16x8(av[u][j], af);
#pragma unroll
        for (int i = 0; i < NW; ++i) {
          float wf[8];
          WC::to_f32(wv[u][i], wf);
          float s = acc[i][j];
#pragma unroll
          for (int e = 0; e < 8; ++e) s = fmaf(af[e], wf[e], s);
          acc[i][j] = s;
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < NW; ++i)
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[i][j] += __shfl_xor_sync(0xffffffffu, acc[i][j], o);
  if (lane == 0) {
    float sc[NW];
#pragma unroll
    for (int i = 0; i < NW; ++i) sc[i] = WT ? __ldg(wscale + wrow_idx[i]) : 1.f;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      if (j >= nr) break;
      __nv_bfloat16* orow = out + static_cast<size_t>(r0 + j) * N + n0;
      if (ACT == 1) {
        const float gt = WT ? acc[0][j] * sc[0] : acc[0][j], up = WT ? acc[1][j] * sc[1] : acc[1][j];
        orow[0] = __float2bfloat16_rn(gt / (1.0f + __expf(-gt)) * up);
      } else {
#pragma unroll
        for (int i = 0; i < NPW; ++i) orow[i] = __float2bfloat16_rn(WT ? acc[i][j] * sc[i] : acc[i][j]);
      }
    }
  }
}

// A one-row SiLU*mul matmul (bf16 weights, one group) that a grouped_gemv
// launch runs before it waits on the previous kernel of its stream: work that
// does not depend on that kernel (the shared expert's gate_up at one token,
// which needs only x).  Only a launch whose predecessor lets dependents start
// after its own wait on its predecessor has returned may carry one (the
// router does so at one token), so that x is complete and `out` is no longer
// read by the call before.
struct GemvPre {
  const __nv_bfloat16* a;   // [1][K]
  const uint8_t* w;         // [2N][K] bf16, gate rows first; nullptr: none
  int N;
  __nv_bfloat16* out;       // [1][N]
};

// (two CTAs per SM: the weight stream needs the loads of 16 warps in flight)
template <int ACT, int R, int WT>
__global__ void __launch_bounds__(kGemvThreads, 2)
    grouped_gemv_kernel(const __nv_bfloat16* __restrict__ a, const uint8_t* __restrict__ w,
                        const float* __restrict__ wscale, const int32_t* __restrict__ offsets, int G, int rows_max,
                        int N, int K, const int32_t* __restrict__ a_rows, int a_src_rows,
                        __nv_bfloat16* __restrict__ out, int* status, const GemvPre pre) {
  constexpr int NPW = ACT == 1 ? 1 : kRowsDown;  // output columns per warp
  __shared__ int s_groups[kMaxGemvGroups];
  __shared__ int s_r0[kMaxGemvGroups], s_nr[kMaxGemvGroups];
  __shared__ int s_src[kMaxGemvGroups * R];      // source rows of a listed group's token rows
  __shared__ int s_count;
  const int warp = threadIdx.x >> 5;
  const long long wstride = static_cast<long long>(gridDim.x) * (kGemvThreads / 32);
  const long long wfirst = static_cast<long long>(blockIdx.x) * (kGemvThreads / 32) + warp;
  if (pre.w)
    for (long long item = wfirst; item < pre.N; item += wstride)
      gemv_item<1, 1, 0>(pre.a, pre.w, nullptr, 0, static_cast<int>(item), 0, 1, pre.N, K, nullptr, 0, 1, pre.out);
  chain_wait();
  const ChainReleaseAtExit release_next;
  list_groups(offsets, G, rows_max, R, status, s_groups, s_r0, s_nr, &s_count);
  // every listed group's source rows, resolved once (one round of loads), so
  // that an item's first memory access is its weight stream
  for (int i = threadIdx.x; i < s_count * R; i += kGemvThreads) {
    const int sl = i / R, j = i - sl * R;
    const int r = s_r0[sl] + (j < s_nr[sl] ? j : s_nr[sl] - 1);
    int src = a_rows ? a_rows[r] : r;
    if (src < 0 || src >= (a_rows ? a_src_rows : rows_max)) src = 0;   // checked upstream; never out of range
    s_src[i] = src;
  }
  __syncthreads();
  const int blocks = N / NPW;                     // output blocks per group
  const long long items = static_cast<long long>(s_count) * blocks;
  for (long long item = wfirst; item < items; item += wstride) {
    const int sl = static_cast<int>(item / blocks);
    const int n0 = static_cast<int>(item % blocks) * NPW;
    gemv_item<ACT, R, WT>(a, w, wscale, s_groups[sl], n0, s_r0[sl], s_nr[sl], N, K, a_rows, a_src_rows, rows_max,
                          out, s_src + sl * R);
  }
}

// One token (T = 1): gmm2 and the combine in one pass.  Slot j of the token
// holds row r_j = inv_perm[j], the one row of group g_j.  A CTA owns kTailCols
// consecutive output columns and warp j slot j: the warp reads its h row once
// and the kTailCols weight rows Wd[g_j][n] (contiguous), with kTailSteps K
// strides of loads in flight, and computes y_j[n] = h[r_j] . Wd[g_j][n] exactly
// as the one-row gmm2 above does (lane-strided fp32 sums over K, the same
// butterfly, rounded to bf16).  Then out[n] = bf16(sum_j w_j * y_j[n] +
// shared[n]) with the fp32 adds in slot order, as the combine takes them: the
// same bits as the two launches, without the round trip of y.
// With shared_w given, the shared expert's down matmul runs here too: warp j
// computes shared[n0 + j] = bf16(hs . Wsd[n0 + j]) over all of K_s exactly as
// the one-row matmul does (lanes striding K, fp32 sums, the same butterfly),
// so the result has the same bits as the standalone launch.
constexpr int kTailCols = 8;
constexpr int kTailSteps = 2;
constexpr int kTailSlots = kGemvThreads / 32;   // one warp per slot

template <int WT>
__global__ void __launch_bounds__(kGemvThreads)
    down_combine_gemv_kernel(const __nv_bfloat16* __restrict__ h, const uint8_t* __restrict__ w,
                             const float* __restrict__ wscale, const int32_t* __restrict__ offsets, int G, int rows,
                             int N, int K, int k,
                             const int32_t* __restrict__ inv_perm, const float* __restrict__ topk_w,
                             const __nv_bfloat16* __restrict__ shared, __nv_bfloat16* __restrict__ out,
                             int* status, const __nv_bfloat16* __restrict__ shared_w,
                             const __nv_bfloat16* __restrict__ shared_h, int K_s) {
  __shared__ int s_group[kTailSlots];            // group holding row r (rows <= k), or -1
  __shared__ float s_y[kTailSlots][kTailCols];   // y_j[n], bf16-rounded
  __shared__ int s_live[kTailSlots];
  __shared__ float s_sh[kTailCols];              // the shared expert's down, column n0 + j from warp j
  __shared__ float s_w[kTailSlots];              // the slots' combine weights
  static_assert(kTailCols == kTailSlots, "one warp per column of the shared expert's down");
  using WC = WeightChunk<WT>;
  chain_wait();
  const ChainReleaseAtExit release_next;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this warp's slot row and weight, loaded beside the offsets (one round)
  const int r_slot = warp < k ? __ldg(inv_perm + warp) : -1;
  const float w_slot = threadIdx.x < k ? __ldg(topk_w + threadIdx.x) : 0.f;
  if (threadIdx.x < kTailSlots) s_group[threadIdx.x] = -1;
  __syncthreads();
  for (int g = threadIdx.x; g < G; g += kGemvThreads) {
    const int lo = __ldg(offsets + g), hi = __ldg(offsets + g + 1);
    const bool bad = lo < 0 || hi < lo || hi > rows || hi - lo > 1;
    if (bad) set_status(status, MOE_ERR_DEVICE_CHECK);
    else if (hi > lo) s_group[lo] = g;
  }
  __syncthreads();
  const int n0 = blockIdx.x * kTailCols;
  const int j = warp;
  if (j < k) {
    const int r = r_slot;
    const int g = (r >= 0 && r < rows) ? s_group[r] : -1;   // a row no group holds adds nothing
    float acc[kTailCols];
#pragma unroll
    for (int c = 0; c < kTailCols; ++c) acc[c] = 0.f;
    if (g >= 0) {
      const __nv_bfloat16* hr = h + static_cast<size_t>(r) * K;
      const uint8_t* wr = w + (static_cast<size_t>(g) * N + n0) * K * WC::kBytes;
      for (int kb = lane * 8; kb < K; kb += 256 * kTailSteps) {
        typename WC::Vec wv[kTailSteps][kTailCols];
        uint4 hv[kTailSteps];
#pragma unroll
        for (int u = 0; u < kTailSteps; ++u) {
          const int k0 = kb + u * 256;
          if (k0 < K) {
            hv[u] = __ldg(reinterpret_cast<const uint4*>(hr + k0));
#pragma unroll
            for (int c = 0; c < kTailCols; ++c) wv[u][c] = WC::load(wr + static_cast<size_t>(c) * K * WC::kBytes, k0);
          }
        }
#pragma unroll
        for (int u = 0; u < kTailSteps; ++u) {
          if (kb + u * 256 >= K) break;
          float af[8];
          bf16x8(hv[u], af);
#pragma unroll
          for (int c = 0; c < kTailCols; ++c) {
            float wf[8];
            WC::to_f32(wv[u][c], wf);
            float s = acc[c];
#pragma unroll
            for (int e = 0; e < 8; ++e) s = fmaf(af[e], wf[e], s);
            acc[c] = s;
          }
        }
      }
#pragma unroll
      for (int c = 0; c < kTailCols; ++c)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], o);
    }
    if (lane == 0) {
      s_live[j] = g >= 0;
#pragma unroll
      for (int c = 0; c < kTailCols; ++c) {
        const float v = WT && g >= 0 ? acc[c] * __ldg(wscale + static_cast<size_t>(g) * N + n0 + c) : acc[c];
        s_y[j][c] = __bfloat162float(__float2bfloat16_rn(v));
      }
    }
  }
  if (shared_w && n0 + warp < N) {
    const __nv_bfloat16* wrow = shared_w + static_cast<size_t>(n0 + warp) * K_s;
    float acc = 0.f;
    // (eight K strides of loads in flight: one pass for K_s = 2048)
    constexpr int kShSteps = 8;
    for (int kb = lane * 8; kb < K_s; kb += 256 * kShSteps) {
      uint4 hv[kShSteps], wv[kShSteps];
#pragma unroll
      for (int u = 0; u < kShSteps; ++u) {
        const int k0 = kb + u * 256;
        if (k0 < K_s) {
          hv[u] = __ldg(reinterpret_cast<const uint4*>(shared_h + k0));
          wv[u] = __ldg(reinterpret_cast<const uint4*>(wrow + k0));
        }
      }
#pragma unroll
      for (int u = 0; u < kShSteps; ++u) {
        if (kb + u * 256 >= K_s) break;
        float af[8], wf[8];
        bf16x8(hv[u], af);
        bf16x8(wv[u], wf);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(af[e], wf[e], acc);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) s_sh[warp] = acc;
  }
  if (threadIdx.x < kTailSlots) s_w[threadIdx.x] = w_slot;
  __syncthreads();
  if (threadIdx.x < kTailCols && n0 + static_cast<int>(threadIdx.x) < N) {
    const int n = n0 + threadIdx.x;
    float v = 0.f;
    for (int s = 0; s < k; ++s)
      if (s_live[s]) v = fmaf(s_w[s], s_y[s][threadIdx.x], v);
    if (shared_w) {
      v += __bfloat162float(__float2bfloat16_rn(s_sh[threadIdx.x]));
    } else if (shared) {
      v += __bfloat162float(shared[n]);
    }
    out[n] = __float2bfloat16_rn(v);
  }
}

}  // namespace

bool down_combine_gemv_applies(int G, int N, int K, int k) {
  return k <= kTailSlots && N % kTailCols == 0 && grouped_gemv_applies(G, N, K, 0, 1);
}

int down_combine_gemv_launch(const void* h, const void* w_down, const float* w_scale, const int32_t* offsets, int G,
                             int N, int K, int k, const int32_t* inv_perm, const float* topk_w, const void* shared,
                             void* out, int* status, cudaStream_t stream, int* launches, const void* shared_w,
                             const void* shared_h, int K_s) {
  if (k < 1 || k > kTailSlots || N % kTailCols) return MOE_ERR_UNSUPPORTED;
  if (shared_w && (!shared_h || K_s <= 0 || K_s % 8)) return MOE_ERR_UNSUPPORTED;
  const dim3 g(N / kTailCols), b(kGemvThreads);
  const cudaError_t rc = launch_chained(
      w_scale ? down_combine_gemv_kernel<1> : down_combine_gemv_kernel<0>, g, b, 0, stream,
      static_cast<const __nv_bfloat16*>(h), static_cast<const uint8_t*>(w_down), w_scale, offsets, G, k, N, K, k,
      inv_perm, topk_w, static_cast<const __nv_bfloat16*>(shared), static_cast<__nv_bfloat16*>(out), status,
      static_cast<const __nv_bfloat16*>(shared_w), static_cast<const __nv_bfloat16*>(shared_h), K_s);
  if (rc != cudaSuccess) return MOE_ERR_CUDA;
  ++*launches;
  return MOE_OK;
}

bool grouped_gemv_applies(int G, int N, int K, int act, int max_group_rows) {
  return max_group_rows == 1 && G <= kMaxGemvGroups && K % 8 == 0 && (act == 1 || N % kRowsDown == 0);
}

int grouped_gemv_launch(const void* a, const void* w, const float* w_scale, const int32_t* offsets, int G,
                        int rows_max, int N, int K, int act, void* out, int* status, cudaStream_t stream,
                        int* launches, const int32_t* a_rows, int a_src_rows, int max_group_rows, int grid_cap,
                        const void* pre_a, const void* pre_w, int pre_N, void* pre_out) {
  if (rows_max == 0 && !pre_w) return MOE_OK;
  // at most min(G, rows_max) non-empty groups
  const long long groups = G < rows_max ? G : rows_max;
  long long items = groups * (act == 1 ? N : N / kRowsDown);
  if (max_group_rows != 1) return MOE_ERR_UNSUPPORTED;
  if (pre_w && (!pre_a || !pre_out || pre_N <= 0)) return MOE_ERR_UNSUPPORTED;
  if (pre_w && pre_N > items) items = pre_N;   // the items of the pre-wait matmul go first, on the same warps
  const int form = (act == 1 ? 1 : 0) + (w_scale ? 2 : 0);
  auto kernel = form == 0 ? grouped_gemv_kernel<0, 1, 0>
                          : form == 1 ? grouped_gemv_kernel<1, 1, 0>
                                      : form == 2 ? grouped_gemv_kernel<0, 1, 1> : grouped_gemv_kernel<1, 1, 1>;
  // persistent: no more CTAs than stay resident (each lists the groups once)
  long long grid = (items + kGemvThreads / 32 - 1) / (kGemvThreads / 32);
  int* dev_status = nullptr;
  int sms = 0;
  static std::atomic<int> occupancy[4] = {};   // resident CTAs per SM of each form (looked up once)
  if (current_device_info(&dev_status, &sms) != MOE_OK) return MOE_ERR_CUDA;
  int per_sm = occupancy[form].load(std::memory_order_relaxed);
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kGemvThreads, 0) != cudaSuccess)
      return MOE_ERR_CUDA;
    occupancy[form].store(per_sm, std::memory_order_relaxed);
  }
  // resident CTAs of the SMs the launch may fill
  const long long resident = static_cast<long long>(grid_cap > 0 && grid_cap < sms ? grid_cap : sms) *
                             (per_sm > 0 ? per_sm : 1);
  if (grid > resident) grid = resident;
  const dim3 g(static_cast<unsigned>(grid)), b(kGemvThreads);
  const GemvPre pre{static_cast<const __nv_bfloat16*>(pre_a), static_cast<const uint8_t*>(pre_w), pre_N,
                    static_cast<__nv_bfloat16*>(pre_out)};
  const cudaError_t rc = launch_chained(kernel, g, b, 0, stream, static_cast<const __nv_bfloat16*>(a),
                                        static_cast<const uint8_t*>(w), w_scale, offsets, G, rows_max, N, K, a_rows,
                                        a_src_rows, static_cast<__nv_bfloat16*>(out), status, pre);
  if (rc != cudaSuccess) return MOE_ERR_CUDA;
  ++*launches;
  return MOE_OK;
}

}  // namespace moe
