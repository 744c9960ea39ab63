// Router pieces of route.cu: the fp32 partial dot products of x with router
// rows over slices of H, the sum of the slices, the warp top-k with its
// softmax over the chosen logits, and the counting sort of a small batch's
// (token, slot) pairs in shared memory.
#pragma once

#include "common.cuh"

namespace moe {

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

constexpr int kSliceH = 512;            // H elements per partial-logit warp
constexpr int kMaxSlices = 8;           // at most this many H slices

__host__ __device__ inline int small_slices(int H) {
  int S = H / kSliceH;
  if (S < 1) S = 1;
  if (S > kMaxSlices) S = kMaxSlices;
  while (S > 1 && H % (S * 8)) --S;
  return S;
}

// One warp: acc[t] = sum over h in [h_begin, h_end) of x[t, h] * w[h] for the
// NT token rows of x (rows at or past nrows re-read row nrows-1, so that every
// load of a step is issued unconditionally); lanes stride h eight elements at
// a time (16-byte loads), then the lanes' sums are added across the warp.
template <int NT>
__device__ __forceinline__ void warp_partial_dot(const __nv_bfloat16* __restrict__ x, int H, int nrows,
                                                 const float* __restrict__ w, int h_begin, int h_end,
                                                 float (&acc)[NT]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t] = 0.f;
#pragma unroll 2
  for (int h0 = h_begin + lane * 8; h0 < h_end; h0 += 256) {
    const float4 w0 = __ldg(reinterpret_cast<const float4*>(w + h0));
    const float4 w1 = __ldg(reinterpret_cast<const float4*>(w + h0 + 4));
    uint4 xv[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t)
      xv[t] = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t < nrows ? t : nrows - 1) * H + h0));
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      float f[8];
      bf16x8_to_f32(xv[t], f);
      float v = acc[t];
      v = fmaf(f[0], w0.x, v); v = fmaf(f[1], w0.y, v); v = fmaf(f[2], w0.z, v); v = fmaf(f[3], w0.w, v);
      v = fmaf(f[4], w1.x, v); v = fmaf(f[5], w1.y, v); v = fmaf(f[6], w1.z, v); v = fmaf(f[7], w1.w, v);
      acc[t] = v;
    }
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
  }
}

// Top-k of one token by one warp: k rounds of a warp arg-max over the E
// logits (larger value wins, equal values go to the lower id); round r's
// winner stays in lane r.  The chosen ids are then ranked by id across lanes
// (ascending order), and w_j = exp(l_j - max) / sum_i exp(l_i - max) over the
// chosen k, the sum taken by a fixed butterfly.  Registers only.
//
// Refinement (logits from the tensor cores, refine != nullptr): if the k-th
// and (k+1)-th logits lie within kRefineDelta (5e-4, at least 8x the
// tensor-core logit error measured at these sizes), every expert whose logit lies
// within kRefineDelta of the k-th is re-evaluated with fp32 FMAs (x . Wr[e] +
// b[e]) and the selection is run again.  The tensor-core logits differ from
// fp32 ones by far less than kRefineDelta / 2, so experts outside that band
// keep their side of the boundary and the choice equals the fp32 choice.
constexpr float kRefineDelta = 5e-4f;

struct Refine {
  const __nv_bfloat16* x;   // this token's row [H]
  const float* wr;          // [E][H]
  int H;
};

__device__ __forceinline__ float warp_dot_fp32(const __nv_bfloat16* x, const float* w, int H) {
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
#pragma unroll 4
  for (int h0 = lane * 8; h0 < H; h0 += 256) {
    const uint4 xv = *reinterpret_cast<const uint4*>(x + h0);
    const float4 w0 = *reinterpret_cast<const float4*>(w + h0);
    const float4 w1 = *reinterpret_cast<const float4*>(w + h0 + 4);
    float f[8];
    bf16x8_to_f32(xv, f);
    acc = fmaf(f[0], w0.x, acc); acc = fmaf(f[1], w0.y, acc); acc = fmaf(f[2], w0.z, acc); acc = fmaf(f[3], w0.w, acc);
    acc = fmaf(f[4], w1.x, acc); acc = fmaf(f[5], w1.y, acc); acc = fmaf(f[6], w1.z, acc); acc = fmaf(f[7], w1.w, acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

// k rounds of arg-max over v (lane-strided, E entries); returns this lane's
// round winner (lane r keeps round r) and the value of round `extra` (-inf if none).
// Order-preserving map of a float to a 32-bit key (a larger float gives a
// larger key; -0 and +0 give the same key).  Key 0 is below every float's key
// (the key of -inf is 0x007fffff) and marks "not a candidate".
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t b = __float_as_uint(v == 0.f ? 0.f : v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// `rounds` rounds of "take the largest remaining logit, the smallest expert
// id among equal values", one warp, lane j keeping round j's (id, value);
// last_v = the value of the final round.  Each round is a lane-local pass over
// the lane's NPL keys and two warp reductions (max key, then min id among
// the lanes holding it).
template <int NPL>
__device__ __forceinline__ void warp_select(const float (&v)[NPL], int E, int rounds, int& my_id, float& my_v,
                                            float& last_v) {
  const int lane = threadIdx.x & 31;
  uint32_t key[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) key[i] = i * 32 + lane < E ? order_key(v[i]) : 0u;
  my_id = 0x7fffffff;
  my_v = -INFINITY;
  last_v = -INFINITY;
  for (int r = 0; r < rounds; ++r) {
    uint32_t bk = 0;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (key[i] > bk) { bk = key[i]; bi = i; }   // strict: equal keys keep the smaller id
    const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
    const int bid = __reduce_min_sync(0xffffffffu, bk == m ? bi * 32 + lane : 0x7fffffff);
    const float best = key_value(m);
    if (lane == r) { my_id = bid; my_v = best; }
    last_v = best;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
      if (i * 32 + lane == bid) key[i] = 0u;
  }
}

// NPL = logits per lane (E <= 32 * NPL).
// S > 1: the logits are S partial slices, slice s at l + s * stride, added in
// slice order (every load issued before the first add).
template <int NPL>
__device__ void warp_topk_softmax(const float* l, const float* bias, int E, int k, int32_t* ids_out, float* w_out,
                                  const Refine* refine = nullptr, int S = 1, size_t stride = 0) {
  const int lane = threadIdx.x & 31;
  float v[NPL];
  if (S == 1) {
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = i * 32 + lane;
      v[i] = e < E ? l[e] + (bias ? bias[e] : 0.f) : -INFINITY;
    }
  } else {
    float p[NPL][kMaxSlices];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = min(i * 32 + lane, E - 1);
#pragma unroll
      for (int sl = 0; sl < kMaxSlices; ++sl) p[i][sl] = l[(sl < S ? sl : S - 1) * stride + e];
    }
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = i * 32 + lane;
      float acc = p[i][0];
#pragma unroll
      for (int sl = 1; sl < kMaxSlices; ++sl)
        if (sl < S) acc += p[i][sl];
      v[i] = e < E ? acc + (bias ? bias[e] : 0.f) : -INFINITY;
    }
  }
  int my_id;
  float my_v, last_v;
  bool selected = false;
  if (refine && k < E) {
    warp_select(v, E, k + 1, my_id, my_v, last_v);   // round k holds the (k+1)-th value
    const float vk = __shfl_sync(0xffffffffu, my_v, k - 1);
    // no near tie: rounds 0..k-1 already are the choice (lane k's extra round is dropped below)
    selected = !(vk - last_v < kRefineDelta);
    if (!selected) {
#pragma unroll
      for (int i = 0; i < NPL; ++i) {
        const int e0 = i * 32;
        if (e0 >= E) break;
        uint32_t band = __ballot_sync(0xffffffffu, e0 + lane < E && fabsf(v[i] - vk) <= kRefineDelta);
        while (band) {
          const int src = __ffs(band) - 1;
          band &= band - 1;
          const int e = e0 + src;
          const float exact = warp_dot_fp32(refine->x, refine->wr + static_cast<size_t>(e) * refine->H, refine->H) +
                              (bias ? bias[e] : 0.f);
          if (lane == src) v[i] = exact;
        }
      }
    }
  }
  if (!selected) warp_select(v, E, k, my_id, my_v, last_v);
  if (lane >= k) { my_id = 0x7fffffff; my_v = -INFINITY; }
  // position of this lane's id among the chosen ids
  int rank = 0;
  for (int j = 0; j < k; ++j) rank += __shfl_sync(0xffffffffu, my_id, j) < my_id ? 1 : 0;
  const float m = __shfl_sync(0xffffffffu, my_v, 0);   // round 0 took the maximum
  const float p = lane < k ? expf(my_v - m) : 0.f;
  float sum = p;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    ids_out[rank] = my_id;
    w_out[rank] = p / sum;
  }
}

// Logit i of a batch from S partial slices part[s * slice + i] (slice =
// T * E): the slices added in slice order, then the bias.  Every load goes
// out before the first add (slices past S re-read slice S-1, not added).
__device__ __forceinline__ float sliced_logit(const float* part, int S, size_t slice, int i, float bias) {
  float p[kMaxSlices];
#pragma unroll
  for (int sl = 0; sl < kMaxSlices; ++sl) p[sl] = __ldcg(part + (sl < S ? sl : S - 1) * slice + i);
  float v = p[0];
#pragma unroll
  for (int sl = 1; sl < kMaxSlices; ++sl)
    if (sl < S) v += p[sl];
  return v + bias;
}

// Counting sort of the T*k pairs of a batch of T <= 32 tokens by (expert,
// token), by one CTA in shared memory: ids[T*k] (slot order per token) ->
// off[E] (exclusive prefix of the counts; *total = T*k), sorted[T*k] (token of
// row r), inv[T*k] (row of pair i).  mask[E] is scratch (one bit per token).
// Every thread of the CTA calls it; nthreads = blockDim.x.
__device__ __forceinline__ void block_sort_small(const int32_t* ids, int T, int k, int E, uint32_t* mask, int* off,
                                                 int* total, int32_t* sorted, int32_t* inv) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < E; e += blockDim.x) mask[e] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) atomicOr(&mask[ids[i]], 1u << (i / k));
  __syncthreads();
  if (warp == 0) {   // exclusive scan of the counts over experts
    int run = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int c = e < E ? __popc(mask[e]) : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      if (e < E) off[e] = run + incl - c;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) *total = run;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
    const int t = i / k, e = ids[i];
    const int r = off[e] + __popc(mask[e] & ((1u << t) - 1u));
    sorted[r] = t;
    inv[i] = r;
  }
  __syncthreads();
}

}  // namespace moe
