// Dispatch of the MoE FFN layer at one expert-parallel rank: a counting sort of
// the T*k (token, slot) pairs by (expert ascending, token ascending), the
// per-expert row offsets of the grouped matmuls, the inverse map used by the
// combine, and the row copy x_perm[r] = x[sorted_token[r]].
//
// "dispatch" is the step before gmm1 on the routed path ("Ascend 910C LLM
// inference optimisation, part 2" (Dewu Tech), section on MoE multi-stream
// overlap); its result stays on the device, as the same page's sampling
// section asks of index work (no device-to-host sync on the path).
//
// Determinism: within a block of 256 tokens, the pairs of expert e form a
// 256-bit mask indexed by token (atomicOr, order-free).  The rank of pair
// (t, e) among the block's pairs of e is the popcount of the mask bits below
// t; adding the block's base (the pairs of e in earlier blocks plus the pairs
// of smaller experts) gives the row.  Nothing depends on thread scheduling.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kTB = 256;            // tokens per block (threads per block)
constexpr int kMaskWords = kTB / 32;

// Token t's k expert ids in registers, every load issued at once (slots past
// k hold -1): one memory round trip instead of one per slot.
__device__ __forceinline__ void load_ids(const int32_t* __restrict__ ids, int t, int k, int (&e)[kMaxTopK]) {
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) e[j] = j < k ? ids[static_cast<size_t>(t) * k + j] : -1;
}

// Validates a token's ids (in [0,E), pairwise distinct) and ORs its bit (local
// token tl) into the block mask.  Returns false (and records the error) for a
// bad token.
__device__ __forceinline__ bool mask_token(const int (&e)[kMaxTopK], int tl, int E, int k, uint32_t* mask,
                                           int* status) {
  bool ok = true;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j < k) {
      if (e[j] < 0 || e[j] >= E) ok = false;
#pragma unroll
      for (int i = 0; i < j; ++i)
        if (e[i] == e[j]) ok = false;
    }
  }
  if (!ok) {
    set_status(status, MOE_ERR_DEVICE_CHECK);
    return false;
  }
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j)
    if (j < k) atomicOr(&mask[e[j] * kMaskWords + (tl >> 5)], 1u << (tl & 31));
  return true;
}

__device__ __forceinline__ int mask_count(const uint32_t* mask, int e) {
  int c = 0;
#pragma unroll
  for (int w = 0; w < kMaskWords; ++w) c += __popc(mask[e * kMaskWords + w]);
  return c;
}

__device__ __forceinline__ int mask_rank(const uint32_t* mask, int e, int tl) {
  int c = 0;
  const int wt = tl >> 5;
  for (int w = 0; w < wt; ++w) c += __popc(mask[e * kMaskWords + w]);
  return c + __popc(mask[e * kMaskWords + wt] & ((1u << (tl & 31)) - 1u));
}

// In-place exclusive scan of v[0..n) (n <= 4 * kTB) by a block of kTB
// threads; returns the total.  Every thread must call it.
__device__ int block_exclusive_scan(int* v, int n) {
  __shared__ int warp_tot[kTB / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n + kTB - 1) / kTB;
  const int i0 = tid * per;
  int local = 0;
  for (int i = 0; i < per; ++i)
    if (i0 + i < n) local += v[i0 + i];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int wbase = 0, total = 0;
  for (int w = 0; w < kTB / 32; ++w) {
    if (w < warp) wbase += warp_tot[w];
    total += warp_tot[w];
  }
  int run = wbase + incl - local;
  for (int i = 0; i < per; ++i)
    if (i0 + i < n) {
      const int c = v[i0 + i];
      v[i0 + i] = run;
      run += c;
    }
  __syncthreads();
  return total;
}

// T <= kTB: the whole sort in one block.
__global__ void __launch_bounds__(kTB)
    permute_small_kernel(const int32_t* __restrict__ ids, int T, int E, int k, int32_t* __restrict__ offsets,
                         int32_t* __restrict__ sorted_token, int32_t* __restrict__ inv_perm, int* status) {
  __shared__ uint32_t mask[kMaxExperts * kMaskWords];
  __shared__ int s_off[kMaxExperts];
  chain_wait();
  const ChainReleaseAtExit release_next;
  const int t = threadIdx.x;
  int ev[kMaxTopK];
  load_ids(ids, t < T ? t : 0, k, ev);
  for (int i = t; i < E * kMaskWords; i += kTB) mask[i] = 0;
  __syncthreads();
  const bool valid = t < T && mask_token(ev, t, E, k, mask, status);
  __syncthreads();
  for (int e = t; e < E; e += kTB) s_off[e] = mask_count(mask, e);
  __syncthreads();
  const int total = block_exclusive_scan(s_off, E);
  for (int e = t; e < E; e += kTB) offsets[e] = s_off[e];
  if (t == 0) offsets[E] = total;
  if (t < T) {
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j >= k) continue;
      if (valid) {
        const int r = s_off[ev[j]] + mask_rank(mask, ev[j], t);
        sorted_token[r] = t;
        inv_perm[static_cast<size_t>(t) * k + j] = r;
      } else {
        inv_perm[static_cast<size_t>(t) * k + j] = -1;
      }
    }
  }
}

// Large T, pass 1: per-block expert counts -> block_counts[b][E].
__global__ void __launch_bounds__(kTB)
    permute_count_kernel(const int32_t* __restrict__ ids, int T, int E, int k, int32_t* __restrict__ block_counts,
                         int* status) {
  __shared__ uint32_t mask[kMaxExperts * kMaskWords];
  chain_wait();
  const ChainReleaseAtExit release_next;
  const int tl = threadIdx.x, t = blockIdx.x * kTB + tl;
  int ev[kMaxTopK];
  load_ids(ids, t < T ? t : 0, k, ev);
  for (int i = tl; i < E * kMaskWords; i += kTB) mask[i] = 0;
  __syncthreads();
  if (t < T) mask_token(ev, tl, E, k, mask, status);
  __syncthreads();
  for (int e = tl; e < E; e += kTB) block_counts[static_cast<size_t>(blockIdx.x) * E + e] = mask_count(mask, e);
}

// Large T, pass 2: rows of every pair of the block.  Each block first derives
// its own bases from the count matrix (every block reads all of it, B x E
// ints): base[e] = offsets[e] + sum over blocks b' < b of counts[b'][e], with
// offsets the exclusive scan of the expert totals; block 0 writes offsets.
__global__ void __launch_bounds__(kTB)
    permute_scatter_kernel(const int32_t* __restrict__ ids, int T, int E, int k,
                           const int32_t* __restrict__ block_counts, int32_t* __restrict__ offsets,
                           int32_t* __restrict__ sorted_token, int32_t* __restrict__ inv_perm) {
  __shared__ uint32_t mask[kMaxExperts * kMaskWords];
  __shared__ int s_tot[kMaxExperts];
  __shared__ int s_before[kMaxExperts];
  chain_wait();
  const ChainReleaseAtExit release_next;
  const int tl = threadIdx.x, t = blockIdx.x * kTB + tl;
  const int b = blockIdx.x, B = gridDim.x;
  int ev[kMaxTopK];
  load_ids(ids, t < T ? t : 0, k, ev);
  for (int i = tl; i < E * kMaskWords; i += kTB) mask[i] = 0;
  for (int e = tl; e < E; e += kTB) {
    int before = 0, tot = 0;
#pragma unroll 8
    for (int bb = 0; bb < B; ++bb) {
      const int c = block_counts[static_cast<size_t>(bb) * E + e];
      tot += c;
      if (bb < b) before += c;
    }
    s_tot[e] = tot;
    s_before[e] = before;
  }
  __syncthreads();
  // errors were recorded by the count pass
  const bool valid = t < T && mask_token(ev, tl, E, k, mask, nullptr);
  const int total = block_exclusive_scan(s_tot, E);   // s_tot -> offsets
  if (b == 0) {
    for (int e = tl; e < E; e += kTB) offsets[e] = s_tot[e];
    if (tl == 0) offsets[E] = total;
  }
  if (t >= T) return;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j >= k) continue;
    if (valid) {
      const int e = ev[j];
      const int r = s_tot[e] + s_before[e] + mask_rank(mask, e, tl);
      sorted_token[r] = t;
      inv_perm[static_cast<size_t>(t) * k + j] = r;
    } else {
      inv_perm[static_cast<size_t>(t) * k + j] = -1;
    }
  }
}

// x_perm[inv_perm[t*k + j]] = x[t]: one warp per token reads its row once (16-byte
// loads) and writes its k copies, so x is read from memory once even when it
// does not fit in L2.  A lane issues the loads of up to kRowChunk of its
// 16-byte pieces before the first store (one memory round trip per 2048
// bf16 of H instead of one per 256).  Pairs the sort rejected (row -1) are
// skipped.
constexpr int kRowChunk = 8;

__global__ void __launch_bounds__(256)
    scatter_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ inv_perm, int T, int H, int k,
                        long long rows_max, uint4* __restrict__ x_perm) {
  chain_wait();
  const ChainReleaseAtExit release_next;
  const int vec = H / 8;
  const int lane = threadIdx.x & 31;
  for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < T; t += gridDim.x * 8) {
    int dst[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      const int r = j < k ? inv_perm[static_cast<size_t>(t) * k + j] : -1;
      dst[j] = (r >= 0 && r < rows_max) ? r : -1;
    }
    const uint4* src = x + static_cast<size_t>(t) * vec;
    for (int i0 = 0; i0 < vec; i0 += 32 * kRowChunk) {
      uint4 v[kRowChunk];
#pragma unroll
      for (int c = 0; c < kRowChunk; ++c) {
        const int i = i0 + c * 32 + lane;
        if (i < vec) v[c] = __ldg(src + i);
      }
#pragma unroll
      for (int c = 0; c < kRowChunk; ++c) {
        const int i = i0 + c * 32 + lane;
        if (i >= vec) continue;
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j)
          if (dst[j] >= 0) x_perm[static_cast<size_t>(dst[j]) * vec + i] = v[c];
      }
    }
  }
}

}  // namespace

size_t permute_ws_bytes(int T, int E) {
  const size_t B = (static_cast<size_t>(T) + kTB - 1) / kTB;
  return T <= kTB ? 0 : align_up(B * E * sizeof(int32_t));
}

int permute_launch(const int32_t* topk_ids, const void* x, int T, int H, int E, int k, int32_t* offsets,
                   int32_t* sorted_token, int32_t* inv_perm, void* x_perm, int32_t* block_counts, int* status,
                   int num_sms, cudaStream_t stream, int* launches) {
  if (T == 0) return MOE_OK;
  if (T <= kTB) {
    if (launch_chained(permute_small_kernel, dim3(1), dim3(kTB), 0, stream, topk_ids, T, E, k, offsets, sorted_token,
                       inv_perm, status) != cudaSuccess)
      return MOE_ERR_CUDA;
    ++*launches;
  } else {
    const int B = (T + kTB - 1) / kTB;
    if (launch_chained(permute_count_kernel, dim3(B), dim3(kTB), 0, stream, topk_ids, T, E, k, block_counts,
                       status) != cudaSuccess ||
        launch_chained(permute_scatter_kernel, dim3(B), dim3(kTB), 0, stream, topk_ids, T, E, k,
                       static_cast<const int32_t*>(block_counts), offsets, sorted_token, inv_perm) != cudaSuccess)
      return MOE_ERR_CUDA;
    *launches += 2;
  }
  if (x_perm) {
    long long grid = (static_cast<long long>(T) + 7) / 8;
    if (grid > 8LL * num_sms) grid = 8LL * num_sms;
    if (launch_chained(scatter_rows_kernel, dim3(static_cast<int>(grid)), dim3(256), 0, stream,
                       static_cast<const uint4*>(x), static_cast<const int32_t*>(inv_perm), T, H, k,
                       static_cast<long long>(T) * k, static_cast<uint4*>(x_perm)) != cudaSuccess)
      return MOE_ERR_CUDA;
    ++*launches;
  }
  return MOE_OK;
}

}  // namespace moe
