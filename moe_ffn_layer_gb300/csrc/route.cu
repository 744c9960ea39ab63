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
// Kernels:
//   T == 1    route_cluster: one 8-CTA cluster, a warp per expert over all of H,
//             the logits gathered in one CTA's shared memory (no ticket).
//   T <= 16   route_small: one warp per (expert, 512-wide slice of H)
//             streams its slice of Wr once and dots it with every token; the
//             CTA that finishes last (a ticket counter) adds the slices in
//             slice order, takes the top-k and, inside the layer forward, runs
//             the counting sort as well.  Decode shapes: one launch.
//   T >  16   logits, then topk_softmax (one warp per token; adds the bias).
//             Logits for T >= 512 (E, H multiples of 64) come from the tensor
//             cores: each fp32 weight is split exactly into three bf16 terms
//             w = hi + mid + lo (hi = bf16(w), mid = bf16(w - hi), lo =
//             bf16(w - hi - mid); every subtraction is exact in fp32 and the
//             three terms carry the full 24-bit significand), and since x is
//             bf16 every product x*term is exact in fp32; the grouped GEMM
//             adds them in fp32 with K = 3H.  Otherwise fp32 FMAs over up
//             to 8 slices of H (the top-k adds the slices in slice order):
//             below 128 tokens one warp per (expert, slice, 16 tokens), from
//             128 tokens a 64 x 64 SIMT tile GEMM per slice.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {
namespace {

// fp32 SIMT GEMM over one slice of H: part[z][T][E] = x[T][hz] . Wr[E][hz]^T
// for the z-th of gridDim.z equal slices hz of H (one slice: the logits).  CTA
// tile 64 x 64, K chunk 32, 256 threads each owning a 4 x 4 block of outputs;
// the next chunk is loaded into registers while the current one is used.
constexpr int kRT = 64, kRE = 64, kRK = 32;

__global__ void __launch_bounds__(256)
    router_tile_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ wr, int T, int H, int E,
                       float* __restrict__ part) {
  __shared__ float xs[kRK][kRT + 4];
  __shared__ float ws[kRK][kRE + 4];
  chain_wait();
  const ChainReleaseAtExit release_next;
  const int t0 = blockIdx.x * kRT, e0 = blockIdx.y * kRE;
  const int HS = H / gridDim.z;
  const int kbeg = blockIdx.z * HS, kend = kbeg + HS;
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;   // 16 x 16 threads
  // this thread's share of a chunk: 8 bf16 of one x row, 2 x 4 fp32 of Wr rows
  const int xr = tid >> 2, xc = (tid & 3) * 8;
  uint4 xv;
  float4 wv[2];
  auto fetch = [&](int k0) {
    xv = make_uint4(0, 0, 0, 0);
    if (t0 + xr < T && k0 + xc < kend)
      xv = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t0 + xr) * H + k0 + xc));
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const int idx = tid + p * 256;
      const int r = idx >> 3, c = (idx & 7) * 4;
      wv[p] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e0 + r < E && k0 + c < kend)
        wv[p] = __ldg(reinterpret_cast<const float4*>(wr + static_cast<size_t>(e0 + r) * H + k0 + c));
    }
  };
  float acc[4][4] = {};
  fetch(kbeg);
  for (int k0 = kbeg; k0 < kend; k0 += kRK) {
    {
      float f[8];
      bf16x8_to_f32(xv, f);
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[xc + i][xr] = f[i];
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int idx = tid + p * 256;
        const int r = idx >> 3, c = (idx & 7) * 4;
        ws[c + 0][r] = wv[p].x; ws[c + 1][r] = wv[p].y; ws[c + 2][r] = wv[p].z; ws[c + 3][r] = wv[p].w;
      }
    }
    __syncthreads();
    if (k0 + kRK < kend) fetch(k0 + kRK);
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
  float* out = part + static_cast<size_t>(blockIdx.z) * T * E;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) out[static_cast<size_t>(t) * E + e] = acc[i][j];
    }
  }
}

// H slices for the tiled router: enough CTAs to cover the GPU, at most
// kMaxSlices, each slice a whole number of K chunks.
int tile_slices(int T, int H, int E, int sms) {
  const int tiles = ((T + kRT - 1) / kRT) * ((E + kRE - 1) / kRE);
  int S = 1;
  while (S < 8 && tiles * S * 2 <= sms && H % (2 * S * kRK) == 0) S *= 2;
  return S;
}

constexpr int kChunkT = 16;             // token rows per partial-logit warp

// 16 < T < 512: partial logits part[s][t][e] over slice s of H, one warp per
// (expert, slice, 16-token chunk); the top-k kernel adds the slices.
__global__ void __launch_bounds__(256)
    router_chunk_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ wr, int T, int H, int E,
                        int S, float* __restrict__ part) {
  chain_wait();
  const ChainReleaseAtExit release_next;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int e = gw % E, sl = (gw / E) % S, t0 = (gw / E / S) * kChunkT;
  if (t0 >= T) return;
  const int nt = min(kChunkT, T - t0);
  const int HS = H / S;
  float acc[kChunkT];
  warp_partial_dot<kChunkT>(x + static_cast<size_t>(t0) * H, H, nt, wr + static_cast<size_t>(e) * H, sl * HS,
                            (sl + 1) * HS, acc);
#pragma unroll
  for (int t = 0; t < kChunkT; ++t)
    if (lane == t && t < nt) part[(static_cast<size_t>(sl) * T + t0 + t) * E + e] = acc[t];
}

// refine_wr != nullptr: the logits came from the tensor cores; near ties are
// re-evaluated in fp32 from x and Wr (see warp_topk_softmax).
// S > 1: logits holds S partial slices [S][T][E], added in slice order.
template <int NPL>
__global__ void __launch_bounds__(256)
    topk_softmax_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int E, int k,
                        int32_t* __restrict__ topk_ids, float* __restrict__ topk_w,
                        const __nv_bfloat16* __restrict__ x, const float* __restrict__ refine_wr, int H, int S) {
  chain_wait();
  const ChainReleaseAtExit release_next;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const Refine r{x + static_cast<size_t>(t) * H, refine_wr, H};
  warp_topk_softmax<NPL>(logits + static_cast<size_t>(t) * E, bias, E, k, topk_ids + static_cast<size_t>(t) * k,
                         topk_w + static_cast<size_t>(t) * k, refine_wr ? &r : nullptr, S,
                         static_cast<size_t>(T) * E);
}

// wr3[e][j*H + h] = j-th bf16 term of Wr[e][h] (j = 0 hi, 1 mid, 2 lo).
__global__ void __launch_bounds__(256)
    split_router_weights_kernel(const float* __restrict__ wr, int E, int H, __nv_bfloat16* __restrict__ wr3) {
  chain_wait();
  const ChainReleaseAtExit release_next;
  const size_t n = static_cast<size_t>(E) * H;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t e = i / H, h = i - e * H;
    const float w = wr[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    __nv_bfloat16* row = wr3 + e * 3 * static_cast<size_t>(H);
    row[h] = hi;
    row[H + h] = mid;
    row[2 * static_cast<size_t>(H) + h] = __float2bfloat16_rn(r2);
  }
}

// ---------------------------------------------------------------- T <= 16: one kernel

constexpr int kSmallT = 16;
constexpr int kSmallThreads = 256;

struct SmallArgs {
  const __nv_bfloat16* x;     // [T][H]
  const float* wr;            // [E][H]
  const float* bias;          // [E] or nullptr
  int T, H, E, k, S;
  float* part;                // [S][T][E] partial logits
  unsigned int* ticket;       // zero on entry; the last CTA sets it back to zero
  int32_t* topk_ids;
  float* topk_w;
  int32_t* offsets;           // nullptr: route only
  int32_t* sorted_token;
  int32_t* inv_perm;
  int early_release;          // let the next kernel start once this one's wait has returned
};

// Every CTA: partial logits part[s][t][e] = sum over slice s of H of
// x[t, h] * Wr[e, h], one warp per (expert, slice), lanes striding the slice
// eight elements at a time (16-byte loads, all of a warp's loads in flight).
// The CTA that arrives last (ticket) adds the slices in slice order (+ bias),
// takes the top-k of every token (one warp per token) and, inside the layer
// forward, runs the counting sort by (expert, token).
// NT: token rows the GEMV carries (a power of two >= T); rows past T re-read
// row T-1, so that every load of a step is issued unconditionally.
template <int NPL, int NT>
__global__ void __launch_bounds__(kSmallThreads) route_small_kernel(const SmallArgs a) {
  __shared__ float logit[kSmallT * kMaxExperts];
  __shared__ int32_t s_ids[kSmallT * kMaxTopK];
  __shared__ float s_w[kSmallT * kMaxTopK];
  __shared__ uint32_t s_mask[kMaxExperts];
  __shared__ int s_off[kMaxExperts];
  __shared__ int s_last, s_total;
  chain_wait();
  // (early release: the previous kernel has completed, so the next one may
  // start its work that depends only on what came before this launch)
  if (a.early_release) chain_release();
  const ChainReleaseAtExit release_next;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = a.T, E = a.E, k = a.k, S = a.S;
  const int gw = blockIdx.x * (kSmallThreads / 32) + warp;
  if (gw < E * S) {
    const int e = gw % E, sl = gw / E;
    const int HS = a.H / S;
    float acc[NT];
    warp_partial_dot<NT>(a.x, a.H, T, a.wr + static_cast<size_t>(e) * a.H, sl * HS, (sl + 1) * HS, acc);
#pragma unroll
    for (int t = 0; t < NT; ++t)
      if (lane == t && t < T) a.part[(static_cast<size_t>(sl) * T + t) * E + e] = acc[t];
  }
  // the last CTA to finish its partials goes on
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(a.ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x == 0) *a.ticket = 0u;   // every CTA has taken its ticket
  const size_t slice = static_cast<size_t>(T) * E;
#pragma unroll 2
  for (int i = threadIdx.x; i < T * E; i += kSmallThreads)
    logit[i] = sliced_logit(a.part, S, slice, i, a.bias ? __ldg(a.bias + i % E) : 0.f);
  __syncthreads();
  for (int t = warp; t < T; t += kSmallThreads / 32)
    warp_topk_softmax<NPL>(logit + t * E, nullptr, E, k, s_ids + t * k, s_w + t * k);
  __syncthreads();
  for (int i = threadIdx.x; i < T * k; i += kSmallThreads) {
    a.topk_ids[i] = s_ids[i];
    a.topk_w[i] = s_w[i];
  }
  if (!a.offsets) return;
  block_sort_small(s_ids, T, k, E, s_mask, s_off, &s_total, a.sorted_token, a.inv_perm);
  for (int e = threadIdx.x; e < E; e += kSmallThreads) a.offsets[e] = s_off[e];
  if (threadIdx.x == 0) a.offsets[E] = s_total;
}

// One token (x small enough for shared memory): one cluster of kClCTAs CTAs
// (16 warps each).  Each warp takes experts w, w + 128, ... (w its index in
// the cluster) and dots each full Wr row with every token: x is staged in
// every CTA's shared memory, Wr is streamed from global memory (a lane's 64
// weights of a 2048-wide chunk of H in flight at once, the warp's first row
// requested before x is staged).  The logits go straight into the first
// CTA's shared memory (distributed shared memory); after the cluster barrier
// that CTA adds the bias, takes the top-k of every token and, in the layer
// forward, runs the counting sort - the same tail as route_small_kernel,
// without the partial-logit round trip through global memory and the ticket.
constexpr int kClCTAs = 8;
constexpr int kClThreads = 512;
constexpr int kClWarps = kClCTAs * kClThreads / 32;
constexpr int kClChunkH = 2048;                 // H per register chunk of a lane (64 fp32 weights)
constexpr int kClLogitBytes = kSmallT * kMaxExperts * 4;
constexpr int kClMaxXBytes = 128 * 1024;        // T * H * 2 at most (else route_small_kernel)

__device__ __forceinline__ void st_cluster_f32(uint32_t local_addr, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

template <int NPL, int NT>
__global__ void __launch_bounds__(kClThreads) route_cluster_kernel(const SmallArgs a) {
  extern __shared__ __align__(16) uint8_t clsm[];
  float* logit = reinterpret_cast<float*>(clsm);                                   // [T][E], CTA 0's is used
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(clsm + kClLogitBytes);     // [T][H]
  __shared__ int32_t s_ids[kSmallT * kMaxTopK];
  __shared__ float s_w[kSmallT * kMaxTopK];
  __shared__ uint32_t s_mask[kMaxExperts];
  __shared__ int s_off[kMaxExperts];
  __shared__ int s_total;
  // every CTA of the cluster has started before any stores into the first
  // one's shared memory: arrive now, wait just before the first such store
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  chain_wait();
  if (a.early_release) chain_release();
  const ChainReleaseAtExit release_next;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = a.T, E = a.E, k = a.k, H = a.H;
  const uint32_t rank = cluster_ctarank();
  const int wfirst = static_cast<int>(rank) * (kClThreads / 32) + warp;
  // a lane's weights of one 2048-wide chunk of a row: h = c + s * 256 + lane * 8 .. + 7, s < 8
  float4 wv[kClChunkH / 256][2];
  auto load_w = [&](int e, int c) {
    const float* row = a.wr + static_cast<size_t>(e) * H + c;
#pragma unroll
    for (int s8 = 0; s8 < kClChunkH / 256; ++s8) {
      const int h = s8 * 256 + lane * 8;
      if (c + h < H) {
        wv[s8][0] = __ldg(reinterpret_cast<const float4*>(row + h));
        wv[s8][1] = __ldg(reinterpret_cast<const float4*>(row + h + 4));
      } else {
        wv[s8][0] = wv[s8][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  };
  if (wfirst < E) load_w(wfirst, 0);
  // x into this CTA's shared memory
  for (int i = threadIdx.x; i < T * H / 8; i += kClThreads)
    reinterpret_cast<uint4*>(xs)[i] = __ldg(reinterpret_cast<const uint4*>(a.x) + i);
  __syncthreads();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  const uint32_t logit_addr = smem_u32(logit);
  for (int e = wfirst; e < E; e += kClWarps) {
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.f;
    for (int c = 0; c < H; c += kClChunkH) {
      if (e != wfirst || c != 0) load_w(e, c);
#pragma unroll
      for (int s8 = 0; s8 < kClChunkH / 256; ++s8) {
        const int h = c + s8 * 256 + lane * 8;
        if (h < H) {
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const int tr = t < T ? t : T - 1;   // rows past T repeat the last (their sums are dropped)
            const uint4 xv = *reinterpret_cast<const uint4*>(xs + static_cast<size_t>(tr) * H + h);
            float f[8];
            bf16x8_to_f32(xv, f);
            float v = acc[t];
            v = fmaf(f[0], wv[s8][0].x, v); v = fmaf(f[1], wv[s8][0].y, v); v = fmaf(f[2], wv[s8][0].z, v);
            v = fmaf(f[3], wv[s8][0].w, v); v = fmaf(f[4], wv[s8][1].x, v); v = fmaf(f[5], wv[s8][1].y, v);
            v = fmaf(f[6], wv[s8][1].z, v); v = fmaf(f[7], wv[s8][1].w, v);
            acc[t] = v;
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
      if (lane == t && t < T) st_cluster_f32(logit_addr + static_cast<uint32_t>((t * E + e) * 4), 0u, acc[t]);
    }
  }
  // every logit has landed in the first CTA (the barrier's release / acquire)
  cluster_sync_all();
  if (rank != 0) return;
  if (a.bias)
    for (int i = threadIdx.x; i < T * E; i += kClThreads) logit[i] += __ldg(a.bias + i % E);
  __syncthreads();
  for (int t = warp; t < T; t += kClThreads / 32)
    warp_topk_softmax<NPL>(logit + t * E, nullptr, E, k, s_ids + t * k, s_w + t * k);
  __syncthreads();
  for (int i = threadIdx.x; i < T * k; i += kClThreads) {
    a.topk_ids[i] = s_ids[i];
    a.topk_w[i] = s_w[i];
  }
  if (!a.offsets) return;
  block_sort_small(s_ids, T, k, E, s_mask, s_off, &s_total, a.sorted_token, a.inv_perm);
  for (int e = threadIdx.x; e < E; e += kClThreads) a.offsets[e] = s_off[e];
  if (threadIdx.x == 0) a.offsets[E] = s_total;
}

template <int NPL>
cudaError_t launch_small_nt(int nt, int grid, cudaStream_t stream, const SmallArgs& a) {
  const dim3 g(grid), b(kSmallThreads);
  switch (nt) {
    case 1: return launch_chained(route_small_kernel<NPL, 1>, g, b, 0, stream, a);
    case 2: return launch_chained(route_small_kernel<NPL, 2>, g, b, 0, stream, a);
    case 4: return launch_chained(route_small_kernel<NPL, 4>, g, b, 0, stream, a);
    case 8: return launch_chained(route_small_kernel<NPL, 8>, g, b, 0, stream, a);
    default: return launch_chained(route_small_kernel<NPL, 16>, g, b, 0, stream, a);
  }
}

// The cluster router's shared-memory attribute, once per (kernel, device).
template <int NPL, int NT>
cudaError_t launch_cluster_one(size_t smem, cudaStream_t stream, const SmallArgs& a) {
  static bool attr_done[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorUnknown;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (dev >= 64 || !attr_done[dev]) {
      const cudaError_t e = cudaFuncSetAttribute(route_cluster_kernel<NPL, NT>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kClLogitBytes + kClMaxXBytes);
      if (e != cudaSuccess) return e;
      if (dev < 64) attr_done[dev] = true;
    }
  }
  return launch_chained_cluster(route_cluster_kernel<NPL, NT>, dim3(kClCTAs), dim3(kClThreads), smem, stream,
                                kClCTAs, a);
}

cudaError_t launch_cluster(int npl, size_t smem, cudaStream_t stream, const SmallArgs& a) {
  if (npl == 4) return launch_cluster_one<4, 1>(smem, stream, a);
  if (npl == 8) return launch_cluster_one<8, 1>(smem, stream, a);
  return launch_cluster_one<16, 1>(smem, stream, a);
}

cudaError_t launch_small(int npl, int nt, int grid, cudaStream_t stream, const SmallArgs& a) {
  if (npl == 4) return launch_small_nt<4>(nt, grid, stream, a);
  if (npl == 8) return launch_small_nt<8>(nt, grid, stream, a);
  return launch_small_nt<16>(nt, grid, stream, a);
}


}  // namespace

constexpr int kTcMinT = 512;   // from this many tokens the logits come from the tensor cores
constexpr int kTileMinT = 128; // from this many tokens (short of that) the tiled fp32 GEMM

bool route_uses_tc(int T, int H, int E) { return T >= kTcMinT && E % 64 == 0 && H % 64 == 0; }

size_t route_ws_bytes(int T, int H, int E) {
  // partial-logit slices: by H for the small and chunked routers, up to
  // kMaxSlices for the tiled one, one for the tensor-core one
  const int slices = T < kTileMinT ? small_slices(H) : (route_uses_tc(T, H, E) ? 1 : kMaxSlices);
  size_t b = align_up(static_cast<size_t>(T) * E * sizeof(float) * slices);
  if (route_uses_tc(T, H, E)) b += align_up(static_cast<size_t>(E) * 3 * H * 2);
  return b;
}

int route_small_max_tokens() { return kSmallT; }

int route_launch(const void* x, const float* w_router, const float* bias, int T, int H, int E, int k,
                 int32_t* topk_ids, float* topk_w, float* logits_ws, unsigned int* ticket, const DispatchOut* dispatch,
                 int* status, int grid_cap, cudaStream_t stream, int* launches, bool early_release) {
  if (T == 0) return MOE_OK;
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  if (T <= kSmallT) {
    if (!ticket) return MOE_ERR_INVALID;
    const int S = small_slices(H);
    const int grid = (E * S + kSmallThreads / 32 - 1) / (kSmallThreads / 32);
    SmallArgs a{xb,      w_router, bias,    T,       H,       E,       k, S, logits_ws, ticket, topk_ids, topk_w,
                nullptr, nullptr,  nullptr, early_release ? 1 : 0};
    if (dispatch) {
      a.offsets = dispatch->offsets;
      a.sorted_token = dispatch->sorted_token;
      a.inv_perm = dispatch->inv_perm;
    }
    const int nt = T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : T <= 8 ? 8 : 16;
    const int npl = E <= 128 ? 4 : E <= 256 ? 8 : 16;
    // one token: the one-cluster router (8 SMs, leaving the rest to the launch
    // that starts beside it); more tokens: the sliced router with its ticket
    // (a warp's full-H dot per token costs more FMAs than the slices save)
    const size_t xbytes = static_cast<size_t>(T) * H * 2;
    if (T == 1 && xbytes <= static_cast<size_t>(kClMaxXBytes) && H % 8 == 0) {
      if (launch_cluster(npl, kClLogitBytes + align_up(xbytes, 16), stream, a) != cudaSuccess)
        return MOE_ERR_CUDA;
    } else if (launch_small(npl, nt, grid, stream, a) != cudaSuccess) {
      return MOE_ERR_CUDA;
    }
    ++*launches;
    return MOE_OK;
  }
  int S = 1;   // partial-logit slices the top-k adds
  if (route_uses_tc(T, H, E)) {
    __nv_bfloat16* wr3 = reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<uint8_t*>(logits_ws) +
                                                          align_up(static_cast<size_t>(T) * E * sizeof(float)));
    const size_t n = static_cast<size_t>(E) * H;
    if (launch_chained(split_router_weights_kernel, dim3(static_cast<int>((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096)),
                       dim3(256), 0, stream, w_router, E, H, wr3) != cudaSuccess)
      return MOE_ERR_CUDA;
    ++*launches;
    const int rc = router_gemm_launch(x, wr3, T, H, E, logits_ws, status, grid_cap, stream, launches);
    if (rc) return rc;
  } else if (T < kTileMinT) {
    S = small_slices(H);
    const long long warps = static_cast<long long>(E) * S * ((T + kChunkT - 1) / kChunkT);
    if (launch_chained(router_chunk_kernel, dim3(static_cast<int>((warps + 7) / 8)), dim3(256), 0, stream, xb,
                       w_router, T, H, E, S, logits_ws) != cudaSuccess)
      return MOE_ERR_CUDA;
    ++*launches;
  } else {
    S = tile_slices(T, H, E, grid_cap);
    dim3 grid((T + kRT - 1) / kRT, (E + kRE - 1) / kRE, S);
    if (launch_chained(router_tile_kernel, grid, dim3(256), 0, stream, xb, w_router, T, H, E, logits_ws) != cudaSuccess)
      return MOE_ERR_CUDA;
    ++*launches;
  }
  const float* rw = route_uses_tc(T, H, E) ? w_router : nullptr;
  const int tg = (T + 7) / 8;
  cudaError_t rc;
  if (E <= 128)
    rc = launch_chained(topk_softmax_kernel<4>, dim3(tg), dim3(256), 0, stream, static_cast<const float*>(logits_ws),
                        bias, T, E, k, topk_ids, topk_w, xb, rw, H, S);
  else if (E <= 256)
    rc = launch_chained(topk_softmax_kernel<8>, dim3(tg), dim3(256), 0, stream, static_cast<const float*>(logits_ws),
                        bias, T, E, k, topk_ids, topk_w, xb, rw, H, S);
  else
    rc = launch_chained(topk_softmax_kernel<16>, dim3(tg), dim3(256), 0, stream, static_cast<const float*>(logits_ws),
                        bias, T, E, k, topk_ids, topk_w, xb, rw, H, S);
  if (rc != cudaSuccess) return MOE_ERR_CUDA;
  ++*launches;
  return MOE_OK;
}

}  // namespace moe
