// GroupedMatmul on the 5th-generation tensor cores (tcgen05 + tensor memory),
// fed by TMA: gmm1 (gate_up, SiLU*mul fused in the epilogue) and gmm2 (down)
// of the routed experts, and the shared expert's two matmuls as one group.
//
// Routed path "dispatch -> gmm1 -> gmm2 -> combine" and the shared expert's
// gate_up/down matmul pair: "Ascend 910C LLM inference optimisation, part 2"
// (Dewu Tech), section on MoE multi-stream overlap.
//
// One persistent, warp-specialised kernel (one CTA per SM) in two tile forms:
//
//  TOKENS_ON_M (prefill; many rows per group): a unit is 128 token rows x BN
//    weight rows.  A = token tile [128 x 64 K], B = weight tile [BN x 64 K]
//    (for SiLU*mul: BN/2 gate rows and the matching BN/2 up rows, so one MMA
//    with N = BN yields both halves in tensor memory).
//  WEIGHTS_ON_M (decode; few rows per group, weight streaming): a unit is 128
//    weight rows x up to NMAX token rows.  A = weight tile [128 x 64 K] (for
//    SiLU*mul: a gate tile and the matching up tile, two MMAs), B = token tile
//    loaded in 16-row boxes, MMA N = token rows rounded up to 16.
//
// Roles:  warp 0      TMA producer into a STAGES-deep shared-memory ring
//         warp 1      tensor-memory allocator and MMA issuer (one thread)
//         warps 2..5  epilogue: tcgen05.ld -> SiLU*mul or identity -> bf16
// The unit list is built on the device from the group offsets (no host sync):
// group g contributes ceil(rows_g / R) x NB units, R = rows per unit, NB =
// weight blocks; empty groups contribute none.  Units are ordered (group,
// weight block, row block) so that CTAs running side by side share a weight
// block in L2.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kBK = 64;            // K per stage: one 128-byte swizzle row of bf16
constexpr int kThreads = 192;      // 6 warps
constexpr int kMaxGroups = 1024;
constexpr int kTileRows128 = 128 * kBK * 2;   // bytes of a 128-row K block
constexpr int kSmemBudget = 200 * 1024;

constexpr int tmem_cols_pow2(int c) { return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : c <= 256 ? 256 : 512; }

// SWAP = 0: tokens on M, W = BN (weight rows per unit).
// SWAP = 1: weights on M, W = NMAX (token rows per unit).
template <int SWAP, int W, int ACT>
struct Cfg {
  static constexpr int kUnitRows = SWAP ? W : 128;                          // token rows per unit
  static constexpr int kABytes = SWAP ? (ACT ? 2 : 1) * kTileRows128 : kTileRows128;
  static constexpr int kBBytes = W * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = kSmemBudget / kStageBytes;
  static constexpr int kOutCols = SWAP ? 128 : (ACT ? W / 2 : W);           // output columns per unit
  static constexpr int kAccCols = SWAP ? (ACT ? 2 : 1) * W : W;             // TMEM columns per unit
  static constexpr int kNumAcc = 2 * kAccCols <= 512 ? 2 : 1;
  static constexpr int kTmemCols = tmem_cols_pow2(kNumAcc * kAccCols);
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 256 + 2 * (kMaxGroups + 1) * 4;
  static_assert(kStages >= 2, "ring too shallow");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

struct GemmArgs {
  const int32_t* offsets;  // [G+1] or nullptr (one group [0, rows_max))
  int G;
  int rows_max;
  int N;                   // output columns
  int K;
  __nv_bfloat16* out;      // [rows_max][N]
  int* status;
  int stream_w;            // weights streamed once: evict-first in L2
};

template <int SWAP, int W, int ACT>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_tok, const __grid_constant__ CUtensorMap tm_wgt,
                        const GemmArgs args) {
  using C = Cfg<SWAP, W, ACT>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_base = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* full_bar = bars;                        // [kStages]
  uint64_t* empty_bar = bars + C::kStages;          // [kStages]
  uint64_t* tfull_bar = bars + 2 * C::kStages;      // [2]
  uint64_t* tempty_bar = tfull_bar + 2;             // [2]
  uint64_t* done_bar = tempty_bar + 2;              // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_total = reinterpret_cast<int*>(tmem_slot + 2);
  int* s_off = reinterpret_cast<int*>(smem + C::kStages * C::kStageBytes + 256);   // [G+1]
  int* s_ustart = s_off + (kMaxGroups + 1);                                          // [G+1]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = args.G;
  const int NB = args.N / C::kOutCols;   // weight blocks per group

  // ---- group table: offsets and unit prefix (warp 0), barriers (warp 1)
  if (warp == 0) {
    const int per = (G + 31) / 32;
    const int g0 = lane * per;
    int local = 0;
    bool bad = false;
    for (int i = 0; i < per; ++i) {
      const int g = g0 + i;
      if (g < G) {
        int a, b;
        if (args.offsets) { a = args.offsets[g]; b = args.offsets[g + 1]; }
        else { a = 0; b = args.rows_max; }
        if (a < 0 || b < a || b > args.rows_max) bad = true;
        s_off[g] = a;
        if (g == G - 1) s_off[G] = b;
        local += ((b - a + C::kUnitRows - 1) / C::kUnitRows) * NB;
      }
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int i = 0; i < per; ++i) {
      const int g = g0 + i;
      if (g < G) {
        s_ustart[g] = run;
        int a, b;
        if (args.offsets) { a = args.offsets[g]; b = args.offsets[g + 1]; }
        else { a = 0; b = args.rows_max; }
        run += ((b - a + C::kUnitRows - 1) / C::kUnitRows) * NB;
      }
    }
    const bool any_bad = __any_sync(0xffffffffu, bad);
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) {
      *s_total = any_bad ? 0 : total;
      *abort_flag = 0;
      if (any_bad && blockIdx.x == 0) set_status(args.status, MOE_ERR_DEVICE_CHECK);
      tma_prefetch_desc(&tm_tok);
      tma_prefetch_desc(&tm_wgt);
    }
  } else if (warp == 1 && lane == 0) {
    for (int s = 0; s < C::kStages; ++s) { mbar_init(&full_bar[s], 1); mbar_init(&empty_bar[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&tfull_bar[b], 1); mbar_init(&tempty_bar[b], 4); }
    mbar_init(done_bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  const int total = *s_total;
  // a CTA without units (or every CTA, when the offsets failed their check)
  // leaves before it allocates tensor memory
  if (static_cast<int>(blockIdx.x) >= total) return;
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // unit index -> group g, first token row, token rows in the unit, weight block
  auto decode = [&](int idx, int& g, int& row0, int& nrows, int& wb) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {                      // last g with ustart[g] <= idx
      const int mid = (lo + hi + 1) >> 1;
      if (s_ustart[mid] <= idx) lo = mid; else hi = mid - 1;
    }
    g = lo;
    const int rows = s_off[g + 1] - s_off[g];
    const int nrb = (rows + C::kUnitRows - 1) / C::kUnitRows;
    const int local = idx - s_ustart[g];
    const int rb = local % nrb;
    wb = local / nrb;
    row0 = s_off[g] + rb * C::kUnitRows;
    nrows = min(rows - rb * C::kUnitRows, C::kUnitRows);
  };

  const int kblocks = args.K / kBK;
  const int wrows = ACT ? 2 * args.N : args.N;   // weight rows per group

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_tok = l2_policy_evict_last();
      const uint64_t pol_w = args.stream_w ? l2_policy_evict_first() : l2_policy_evict_normal();
      long long issued = 0;
      int stage = 0;
      uint32_t phase = 0;
      for (int idx = blockIdx.x; idx < total; idx += gridDim.x) {
        int g, row0, nrows, wb;
        decode(idx, g, row0, nrows, wb);
        const int wrow = g * wrows + wb * C::kOutCols;
        const int n16 = (nrows + 15) >> 4;
        const uint32_t bytes = SWAP ? static_cast<uint32_t>(C::kABytes + n16 * 16 * kBK * 2)
                                    : static_cast<uint32_t>(C::kStageBytes);
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, args.status)) { ok = false; break; }
          uint8_t* sa = stage_base + stage * C::kStageBytes;
          uint8_t* sb = sa + C::kABytes;
          const int kc = kb * kBK;
          mbar_arrive_expect_tx(&full_bar[stage], bytes);
          if (SWAP) {
            tma_load_2d(sa, &tm_wgt, &full_bar[stage], kc, wrow, pol_w);
            if (ACT) tma_load_2d(sa + kTileRows128, &tm_wgt, &full_bar[stage], kc, wrow + args.N, pol_w);
            for (int j = 0; j < n16; ++j)
              tma_load_2d(sb + j * 16 * kBK * 2, &tm_tok, &full_bar[stage], kc, row0 + 16 * j, pol_tok);
          } else {
            tma_load_2d(sa, &tm_tok, &full_bar[stage], kc, row0, pol_tok);
            if (ACT) {
              tma_load_2d(sb, &tm_wgt, &full_bar[stage], kc, wrow, pol_w);
              tma_load_2d(sb + (W / 2) * kBK * 2, &tm_wgt, &full_bar[stage], kc, wrow + args.N, pol_w);
            } else {
              tma_load_2d(sb, &tm_wgt, &full_bar[stage], kc, wrow, pol_w);
            }
          }
          ++issued;
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      // drain: every load issued into the ring has landed before the CTA may
      // exit (bounded wait that ignores `abort`; the normal path passes at once)
      for (int s = 0; s < C::kStages; ++s) {
        const long long fills = issued / C::kStages + (s < issued % C::kStages ? 1 : 0);
        if (fills > 0) mbar_wait_timed(&full_bar[s], static_cast<uint32_t>((fills - 1) & 1), args.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int idx = blockIdx.x; idx < total; idx += gridDim.x, ++it) {
        const int ab = C::kNumAcc == 2 ? (it & 1) : 0;
        const uint32_t aphase = (C::kNumAcc == 2 ? (it >> 1) : it) & 1;
        uint32_t idesc;
        if (SWAP) {
          int g, row0, nrows, wb;
          decode(idx, g, row0, nrows, wb);
          idesc = idesc_bf16_f32(128, ((nrows + 15) >> 4) * 16);
        } else {
          idesc = idesc_bf16_f32(128, W);
        }
        if (!mbar_wait(&tempty_bar[ab], aphase ^ 1u, abort_flag, args.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + ab * C::kAccCols;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abort_flag, args.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(stage_base + stage * C::kStageBytes);
          const uint32_t sb = sa + C::kABytes;
          const uint64_t da = smem_desc_k128(sa);
          const uint64_t db = smem_desc_k128(sb);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // +32 bytes per 16-element K step inside the 128-byte swizzle row
            const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
            umma_bf16(d_tmem, da + static_cast<uint64_t>(kk * 2), db + static_cast<uint64_t>(kk * 2), idesc, acc);
            if (SWAP && ACT) {
              const uint64_t du = smem_desc_k128(sa + kTileRows128);
              umma_bf16(d_tmem + W, du + static_cast<uint64_t>(kk * 2), db + static_cast<uint64_t>(kk * 2), idesc,
                        acc);
            }
          }
          umma_commit(&empty_bar[stage]);      // frees the smem stage when these MMAs finish
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&tfull_bar[ab]);           // accumulator ab ready for the epilogue
      }
      // every MMA issued above has completed once done_bar flips
      umma_commit(done_bar);
      mbar_wait_timed(done_bar, 0, args.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                    // TMEM lane quadrant of this warp
    const int lrow = q * 32 + lane;            // TMEM lane = accumulator row
    int it = 0;
    for (int idx = blockIdx.x; idx < total; idx += gridDim.x, ++it) {
      const int ab = C::kNumAcc == 2 ? (it & 1) : 0;
      const uint32_t aphase = (C::kNumAcc == 2 ? (it >> 1) : it) & 1;
      int g, row0, nrows, wb;
      decode(idx, g, row0, nrows, wb);
      if (!mbar_wait(&tfull_bar[ab], aphase, abort_flag, args.status)) break;
      tc_fence_after();
      const uint32_t t_acc = tmem_base + ab * C::kAccCols + (static_cast<uint32_t>(q * 32) << 16);
      if (SWAP) {
        // accumulator row = output column wb*128 + lrow; accumulator column = token
        __nv_bfloat16* ocol = args.out + static_cast<size_t>(row0) * args.N + wb * 128 + lrow;
#pragma unroll 1
        for (int c = 0; c < nrows; c += 32) {
          uint32_t gr[32];
          tmem_ld_32cols(t_acc + c, gr);
          if (ACT) {
            uint32_t ur[32];
            tmem_ld_32cols(t_acc + W + c, ur);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float gv = __uint_as_float(gr[i]);
              gr[i] = __float_as_uint(gv / (1.0f + __expf(-gv)) * __uint_as_float(ur[i]));
            }
          } else {
            tmem_ld_wait();
          }
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (c + i < nrows) ocol[static_cast<size_t>(c + i) * args.N] = __float2bfloat16_rn(__uint_as_float(gr[i]));
        }
      } else {
        // accumulator row = token row0 + lrow; accumulator column = output column
        const bool live = lrow < nrows;
        __nv_bfloat16* orow = args.out + static_cast<size_t>(row0 + lrow) * args.N + wb * C::kOutCols;
        if (ACT) {
#pragma unroll 1
          for (int c = 0; c < W / 2; c += 32) {
            uint32_t gr[32], ur[32];
            tmem_ld_32cols(t_acc + c, gr);
            tmem_ld_32cols(t_acc + W / 2 + c, ur);
            tmem_ld_wait();
            if (live) {
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float g0 = __uint_as_float(gr[2 * i]), g1 = __uint_as_float(gr[2 * i + 1]);
                const float u0 = __uint_as_float(ur[2 * i]), u1 = __uint_as_float(ur[2 * i + 1]);
                pk[i] = pack_bf16x2(g0 / (1.0f + __expf(-g0)) * u0, g1 / (1.0f + __expf(-g1)) * u1);
              }
              uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
              for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
          }
        } else {
#pragma unroll 1
          for (int c = 0; c < W; c += 32) {
            uint32_t r[32];
            tmem_ld_32cols(t_acc + c, r);
            tmem_ld_wait();
            if (live) {
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
              uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
              for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[ab]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D bf16 tensor [rows][cols] (cols contiguous), box [box_rows][64], 128-byte
// swizzle; loads past the last row read zeros.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int SWAP, int W, int ACT>
int launch_cfg(const void* a, const void* w, const int32_t* offsets, int G, int rows_max, int N, int K, void* out,
               int* status, int grid_cap, cudaStream_t stream, int* launches) {
  using C = Cfg<SWAP, W, ACT>;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !attr_done[dev]) {
    if (cudaFuncSetAttribute(grouped_gemm_kernel<SWAP, W, ACT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (dev < 64) attr_done[dev] = true;
  }
  CUtensorMap tt, tw;
  const int wrows = ACT ? 2 * N : N;
  const uint32_t tok_box = SWAP ? 16 : 128;
  const uint32_t wgt_box = SWAP ? 128 : (ACT ? W / 2 : W);
  if (!make_map(&tt, a, static_cast<uint64_t>(rows_max), static_cast<uint64_t>(K), tok_box)) return MOE_ERR_CUDA;
  if (!make_map(&tw, w, static_cast<uint64_t>(G) * wrows, static_cast<uint64_t>(K), wgt_box)) return MOE_ERR_CUDA;
  // upper bound on the unit count: every non-empty group adds at most one partial row block
  const long long nonempty = offsets ? (G < rows_max ? G : rows_max) : 1;
  const long long bound =
      (static_cast<long long>((rows_max + C::kUnitRows - 1) / C::kUnitRows) + nonempty) * (N / C::kOutCols);
  int grid = static_cast<int>(bound < grid_cap ? bound : grid_cap);
  if (grid < 1) grid = 1;
  const int stream_w = SWAP ? 1 : 0;
  GemmArgs args{offsets, G, rows_max, N, K, reinterpret_cast<__nv_bfloat16*>(out), status, stream_w};
  grouped_gemm_kernel<SWAP, W, ACT><<<grid, kThreads, C::kSmemBytes, stream>>>(tt, tw, args);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  ++*launches;
  return MOE_OK;
}

}  // namespace

bool grouped_gemm_weights_on_m(int G, int rows_max, int N) {
  return N % 128 == 0 && static_cast<long long>(rows_max) <= 64LL * G;
}

int grouped_gemm_launch(const void* a, const void* w, const int32_t* offsets, int G, int rows_max, int N, int K,
                        int act, void* out, int* status, int grid_cap, cudaStream_t stream, int* launches) {
  if (rows_max == 0) return MOE_OK;
  if (grouped_gemm_weights_on_m(G, rows_max, N)) {
    if (act == 1) return launch_cfg<1, 64, 1>(a, w, offsets, G, rows_max, N, K, out, status, grid_cap, stream, launches);
    return launch_cfg<1, 64, 0>(a, w, offsets, G, rows_max, N, K, out, status, grid_cap, stream, launches);
  }
  if (act == 1) {
    if (N % 128 == 0) return launch_cfg<0, 256, 1>(a, w, offsets, G, rows_max, N, K, out, status, grid_cap, stream, launches);
    return launch_cfg<0, 128, 1>(a, w, offsets, G, rows_max, N, K, out, status, grid_cap, stream, launches);
  }
  if (N % 256 == 0) return launch_cfg<0, 256, 0>(a, w, offsets, G, rows_max, N, K, out, status, grid_cap, stream, launches);
  if (N % 128 == 0) return launch_cfg<0, 128, 0>(a, w, offsets, G, rows_max, N, K, out, status, grid_cap, stream, launches);
  return launch_cfg<0, 64, 0>(a, w, offsets, G, rows_max, N, K, out, status, grid_cap, stream, launches);
}

int grouped_gemm_max_groups() { return kMaxGroups; }

}  // namespace moe
