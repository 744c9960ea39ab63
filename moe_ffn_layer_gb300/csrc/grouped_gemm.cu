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
//    loaded in 16-row boxes, MMA N = token rows rounded up to 16.  The K steps
//    go round-robin to up to 4 accumulator chains: an MMA this small is cheap,
//    but one that adds into the accumulator of the MMA just before it waits
//    for it, which would cap the weight stream of an SM far below HBM speed.
//
// Tokens-on-M launches with an even number of 256-wide weight blocks run as
// clusters of two CTAs that load one shared operand tile half each and
// multicast it to both: two 128-row tiles of a group share the weight block,
// an odd last tile is shared by two adjacent weight blocks.  A ring stage is
// released once both CTAs' MMAs are done with it.
//
// Groups of one row never reach this kernel: they run on the CUDA cores
// (gemv.cu), a pure weight stream.
//
// Roles:  warp 0      TMA producer into a STAGES-deep shared-memory ring
//         warp 1      tensor-memory allocator and MMA issuer (one thread)
//         warps 2..5  epilogue: tcgen05.ld -> SiLU*mul or identity -> bf16
// With e4m3 weights (weights-on-M only) warp 0 streams the 8-bit tiles into
// their own ring, warps 6..13 widen them to bf16 in tensor memory (the MMA's A
// operand), warp 14 loads the token tiles into a ring of their own, and the
// epilogue multiplies each row by its scale.  Measured on GB300: one thread
// issues a 128 x 16 x 16 MMA at best every ~50 cycles (two issuing threads
// reach the tensor pipe's ~39), and with its barrier waits and commits the
// issuer needs ~1,400 cycles per 64-wide K step of a gate/up tile pair; so at
// decode sizes the 8-bit stream runs at the MMA issue rate, not at HBM speed.
// The unit list is built on the device from the group offsets (no host sync):
// group g contributes ceil(rows_g / R) x NB units, R = rows per unit, NB =
// weight blocks; empty groups contribute none.  Units are ordered (group,
// weight block, row block) so that CTAs running side by side share a weight
// block in L2.
//
// Leading phase (weights-on-M, bf16): a launch may first compute one group of
// up to 16 token rows with operands of its own (a shared expert), with its own
// split plan and scratch; when those operands do not come from the previous
// kernel it runs before the launch's wait on that kernel.
//
// Stream-K (weights-on-M form, every group <= 16 rows, scratch given; gate_up
// and 8-bit launches): when whole units do not spread evenly over the grid,
// the units' K blocks are laid
// end to end and every CTA takes an equal contiguous share.  A unit cut
// between CTAs becomes pieces; each piece stores its fp32 partial accumulator
// and takes a ticket on the unit's counter; the ticket holder that arrives
// last adds the pieces' partials in piece order, resets the counter to zero
// and runs the epilogue.  The result does not depend on which CTA arrives
// last, and no CTA waits for another.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kBK = 64;            // K per stage: one 128-byte swizzle row of bf16
constexpr int kMaxGroups = 1024;
constexpr int kTileRows128 = 128 * kBK * 2;   // bytes of a 128-row K block
constexpr int kSmemBudget = 216 * 1024;

constexpr int tmem_cols_pow2(int c) { return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : c <= 256 ? 256 : 512; }

// SWAP = 0: tokens on M, W = BN (weight rows per unit).
// SWAP = 1: weights on M, W = NMAX (token rows per unit).
// MC = 1 (tokens-on-M, 256-wide weight blocks): CTAs run in clusters of two
// that share one operand tile, each loading half of it with a multicast to
// both.  A group's 128-row tiles go in twos: the two tiles of a pair share the
// weight block (each CTA loads its own token rows and half of the weights);
// an odd last tile is shared by two adjacent weight blocks instead (each CTA
// loads its own weights and 64 of the tile's token rows).
//
// WT = 1 (weights-on-M only): the weights are e4m3 codes with one fp32 scale
// per weight row.  The producer streams the 8-bit weight tiles into a deep
// ring of their own (the bytes in flight from HBM), limited by nothing but
// that ring; eight converter warps widen each 8-bit tile to bf16 (exact: every
// e4m3 value is a bf16 value) straight into tensor memory, where the MMA reads
// its A operand (a ring of kStages A stages beside the accumulators); a token
// producer warp loads each stage's token tile into the slot of the same index
// (tokens come from L2), and the converters arrive on a stage once its tokens
// have landed too, so the MMA thread waits once and commits once per stage;
// the epilogue multiplies each accumulator row by its scale.
constexpr int kConvWarps = 8;
template <int SWAP, int W, int ACT, int MC = 0, int WT = 0>
struct Cfg {
  // 6 warps (+ the converter warps and the token producer warp)
  static constexpr int kThreads = WT ? 192 + 32 * (kConvWarps + 1) : 192;
  static constexpr int kUnitRows = SWAP ? W : 128;                          // token rows per unit
  static constexpr int kABytes = SWAP ? (ACT == 1 ? 2 : 1) * kTileRows128 : kTileRows128;   // per K block
  // weights-on-M: a stage spans kKB 64-wide K blocks (one MMA-thread wait and
  // commit per kKB * 4 K steps: the small-N MMAs' issue thread is the bound)
  static constexpr int kKB = SWAP ? 2 : 1;
  static constexpr int kBBytes = kKB * W * kBK * 2;                        // token tile(s) of a stage
  // WT: A in tensor memory, tokens apart; else A tiles of the stage's K blocks, then their token tiles
  static constexpr int kStageBytes = WT ? 0 : kKB * kABytes + kBBytes;
  static constexpr int kStages = WT ? (ACT == 1 ? 2 : 4) : kSmemBudget / kStageBytes;   // operand stages
  static constexpr int kTokStages = WT ? kStages : 0;                      // WT: one token slot per A stage
  // WT: 8-bit weights of a stage: 128 rows x kKB * 64 codes per tile (128-byte rows: the DRAM
  // reads of a weight row come in 128-byte runs, as in the bf16 form)
  static constexpr int k8Row = kKB * kBK;
  static constexpr int k8Bytes = WT ? (ACT == 1 ? 2 : 1) * 128 * k8Row : 0;
  static constexpr int k8Stages =
      WT ? (kSmemBudget - kStages * kStageBytes - kTokStages * kBBytes) / k8Bytes : 0;
  static constexpr int kRingBytes = kStages * kStageBytes + kTokStages * kBBytes + k8Stages * k8Bytes;
  static constexpr int kOutCols = SWAP ? 128 : (ACT == 1 ? W / 2 : W);           // output columns per unit
  static constexpr int kAccCols = SWAP ? (ACT == 1 ? 2 : 1) * W : W;             // TMEM columns per unit
  static constexpr int kNumAcc = 2 * kAccCols <= 512 ? 2 : 1;
  // WT: tensor-memory columns of one A stage (128 rows x kKB * 64 bf16 per tile), after the accumulators
  static constexpr int kACols = WT ? (ACT == 1 ? 2 : 1) * kKB * kBK / 2 : 0;
  static constexpr int kAColBase = kNumAcc * kAccCols;
  static constexpr int kTmemCols = tmem_cols_pow2(kAColBase + kStages * kACols);
  // after the rings: the mbarriers (full/empty per stage, 2 tfull, 2 tempty,
  // done; with WT full/empty per 8-bit stage and a token barrier per operand
  // stage), the TMEM slot, the abort flag, the unit total and 8 split words
  static constexpr int kCtrlUsed = (2 * kStages + 6 + 2 * k8Stages + kTokStages) * 8 + 4 + 4 + 4 + 8 * 4;
  static constexpr int kCtrlBytes = (kCtrlUsed + 127) / 128 * 128;
  // the carve, from the 1024-aligned base: operand ring | token ring | 8-bit ring | control | group arrays
  static constexpr int kOffTok = kStages * kStageBytes;
  static constexpr int kOffW8 = kOffTok + kTokStages * kBBytes;
  static constexpr int kOffCtrl = kRingBytes;
  static constexpr int kOffArrays = kRingBytes + kCtrlBytes;
  static constexpr int kArrayBytes = 2 * (kMaxGroups + 1) * 4 + 128 * 4;
  static constexpr int kSmemBytes = 1024 + kOffArrays + kArrayBytes;
  static_assert(kStages >= 2, "ring too shallow");
  static_assert(!WT || (SWAP && !MC && k8Stages >= kTokStages), "8-bit weights: weights-on-M, a deep 8-bit ring");
  static_assert(!WT || kAColBase + kStages * kACols <= 512, "8-bit weights: A stages beside the accumulators");
  static_assert(!WT || k8Row == 2 * kBK, "8-bit weights: one 128-byte box row per stage (make_map_u8)");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

constexpr int kSplitRows = 16;     // split-K only when every group has <= 16 rows
constexpr int kBM_rows = 128;      // token rows of a tokens-on-M unit
constexpr int kMaxSplit = 8;

struct GemmArgs {
  const int32_t* offsets;  // [G+1] or nullptr (one group [0, rows_max))
  int G;
  int rows_max;
  int N;                   // output columns
  int K;
  __nv_bfloat16* out;      // [rows_max][N]
  int* status;
  int stream_w;            // weights streamed once: evict-first in L2
  int* counters;           // split-K tickets, one per unit, zero between calls (nullptr: no split)
  float* partials;         // split-K partial accumulators, split_cap slots
  int split_cap;           // sub-units the scratch holds
  int unit_cap;            // units the counters cover
  int a_kblocks;           // > 0: A has this many K blocks and is re-read for every
                           // run of them along B's K (tokens-on-M form only)
  const int32_t* a_rows;   // non-null: token row r is row a_rows[r] of the token tensor
                           // (fetched with TMA gather4; no permuted copy needed)
  uint64_t wait_ns;        // limit of every bounded wait but the drains (0: expire at once)
  const float* wscale;     // 8-bit weights: one scale per weight row ([G][rows of W[g]])
  // a leading phase (weights-on-M, bf16): one group of pre_rows <= 16 token rows
  // with operands of its own (tensor maps tm_tok2 / tm_wgt2), K = pre_K, output
  // pre_out [pre_rows][pre_N], split-K scratch of its own; pre_early: it runs
  // before the kernel waits on the previous one (its operands do not come from it)
  int pre_units;           // 0: no leading phase
  int pre_N, pre_K, pre_rows, pre_early;
  __nv_bfloat16* pre_out;
  int* pre_counters;       // >= pre_units tickets, zero between calls (nullptr: no split)
  float* pre_partials;
  int pre_split_cap;
};

// A phase of a launch: its units, K blocks and split plan; pre = the leading phase.
struct Phase {
  int mode, S, P, units, kblocks;
  bool pre;
};

// fp32 values one TMEM lane keeps per split-K partial
template <int ACT>
constexpr int partial_floats() { return (ACT == 1 ? 2 : 1) * kSplitRows; }

__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Weights-on-M form: K steps are spread over C independent accumulator chains
// (chain = K step mod C) so that consecutive small-N MMAs do not wait on one
// another; the epilogue adds the chains in order.  C is the largest of 4, 2, 1
// whose chains fit the unit's tensor-memory columns.
__host__ __device__ constexpr int swap_chains(int n16, int acc_cols, int act) {
  return 4 * (act ? 2 : 1) * n16 * 16 <= acc_cols ? 4 : (2 * (act ? 2 : 1) * n16 * 16 <= acc_cols ? 2 : 1);
}

// Work of one CTA as a list of pieces: a piece is K blocks [kb0, kb1) of unit
// u, the pi-th of the np pieces that unit is cut into.
//  mode 0: every unit cut into S equal K ranges (S = 1: whole units); CTA c
//          takes pieces c, c + grid, c + 2 grid, ... of the unit-major list.
//  mode 1 (stream-K): the units' K blocks laid end to end, CTA c takes blocks
//          [c*total/grid, (c+1)*total/grid); a unit cut between CTAs becomes
//          several pieces.
// A unit of np > 1 pieces is finished by whichever piece arrives last.
struct Piece {
  int u, kb0, kb1, pi, np;
};

struct WorkIter {
  int mode, S, units, kblocks, grid, cta;
  long long cur, end, total;
  __device__ static long long start_of(int c, long long total, int grid) {
    return static_cast<long long>(c) * total / grid;
  }
  __device__ int cta_of(long long kk) const {   // CTA whose range holds K block kk
    int c = static_cast<int>(kk * grid / total);
    while (c + 1 < grid && start_of(c + 1, total, grid) <= kk) ++c;
    while (c > 0 && start_of(c, total, grid) > kk) --c;
    return c;
  }
  __device__ WorkIter(int mode_, int S_, int units_, int kblocks_, int grid_, int cta_)
      : mode(mode_), S(S_), units(units_), kblocks(kblocks_), grid(grid_), cta(cta_) {
    total = static_cast<long long>(units) * kblocks;
    if (mode == 0) {
      cur = cta;
      end = static_cast<long long>(units) * S;
    } else {
      cur = start_of(cta, total, grid);
      end = start_of(cta + 1, total, grid);
    }
  }
  __device__ bool empty() const { return cur >= end; }
  __device__ bool next(Piece& p) {
    if (cur >= end) return false;
    if (mode == 0) {
      const int u = static_cast<int>(cur / S), sp = static_cast<int>(cur - static_cast<long long>(u) * S);
      const int per = kblocks / S;
      p = Piece{u, sp * per, (sp + 1) * per, sp, S};
      cur += grid;
      return true;
    }
    const int u = static_cast<int>(cur / kblocks);
    const int kb0 = static_cast<int>(cur - static_cast<long long>(u) * kblocks);
    const long long left = end - cur;
    const int kb1 = left < kblocks - kb0 ? kb0 + static_cast<int>(left) : kblocks;
    const int first = cta_of(static_cast<long long>(u) * kblocks);
    const int last = cta_of(static_cast<long long>(u) * kblocks + kblocks - 1);
    p = Piece{u, kb0, kb1, cta - first, last - first + 1};
    cur += kb1 - kb0;
    return true;
  }
};

// Cost of a piece beyond its K blocks (epilogue, partial store, ticket, the
// last arriver's sum), in K blocks; measured on decode shapes.
constexpr int kPieceCost = 6;

// Split plan of a phase whose groups all hold <= kSplitRows rows: the cheapest
// of S-way splits (S = 1, 2, 4, 8) and (streamk) stream-K, costed as the
// longest CTA's K blocks plus kPieceCost per piece it runs; P = the most
// pieces one unit can be cut into.
__device__ void choose_split(int units, int kblocks, int grid, long long split_cap, bool streamk, int& mode, int& S,
                             int& P) {
  mode = 0;
  S = 1;
  P = 1;
  long long best = static_cast<long long>((units + grid - 1) / grid) * (kblocks + kPieceCost);
  for (int c = 2; c <= kMaxSplit; c *= 2) {
    if (kblocks % c || static_cast<long long>(units) * c > split_cap) continue;
    const long long cost = ((static_cast<long long>(units) * c + grid - 1) / grid) * (kblocks / c + kPieceCost);
    if (cost < best) { best = cost; S = c; P = c; }
  }
  const long long tot = static_cast<long long>(units) * kblocks;
  const long long share = tot / grid;
  if (streamk && share >= 1) {
    const int psk = static_cast<int>((kblocks + share - 1) / share) + 1;
    const long long pieces_per_cta = (share + kblocks - 1) / kblocks + 1;
    const long long cost = (tot + grid - 1) / grid + kPieceCost * pieces_per_cta;
    if (cost < best && static_cast<long long>(units) * psk <= split_cap) {
      mode = 1;
      S = 1;
      P = psk;
    }
  }
}

template <int SWAP, int W, int ACT, int MC = 0, int WT = 0>
__global__ void __launch_bounds__(Cfg<SWAP, W, ACT, MC, WT>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_tok, const __grid_constant__ CUtensorMap tm_wgt,
                        const __grid_constant__ CUtensorMap tm_tok2, const __grid_constant__ CUtensorMap tm_wgt2,
                        const GemmArgs args) {
  static_assert(!MC || (!SWAP && W == 256 && (ACT == 0 || ACT == 1)), "pairs: tokens-on-M, 256-wide blocks");
  constexpr int kTokHalf = 64 * kBK * 2;   // bytes of 64 token rows of a K block
  using C = Cfg<SWAP, W, ACT, MC, WT>;
  constexpr int kThreads = C::kThreads;
  constexpr uint16_t kPairMask = 0x3;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_base = smem;
  uint8_t* tok_base = smem + C::kOffTok;             // token-tile ring (WT)
  uint8_t* w8_base = smem + C::kOffW8;               // 8-bit weight ring (WT)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffCtrl);
  uint64_t* full_bar = bars;                        // [kStages]
  uint64_t* empty_bar = bars + C::kStages;          // [kStages]
  uint64_t* tfull_bar = bars + 2 * C::kStages;      // [2]
  uint64_t* tempty_bar = tfull_bar + 2;             // [2]
  uint64_t* done_bar = tempty_bar + 2;              // [1]
  uint64_t* w8full_bar = done_bar + 1;              // [k8Stages]: 8-bit tile landed
  uint64_t* w8empty_bar = w8full_bar + C::k8Stages; // [k8Stages]: converted
  uint64_t* tokfull_bar = w8empty_bar + C::k8Stages;   // [kTokStages]: token tile landed (freed with its A stage)
  uint64_t* table_bar = tokfull_bar + C::kTokStages;  // [1]: unit table built (after a leading phase)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(table_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_total = reinterpret_cast<int*>(tmem_slot + 2);
  int* s_split = reinterpret_cast<int*>(tmem_slot + 3);   // [0] mode, [1] last arriver, [2..5] warp ok, [6] P, [7] S
  int* s_off = reinterpret_cast<int*>(smem + C::kOffArrays);                       // [G+1]
  int* s_ustart = s_off + (kMaxGroups + 1);                                          // [G+1]
  int* s_gidx = s_ustart + (kMaxGroups + 1);                                         // [128] gathered rows

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = args.G;
  const int NB = args.N / C::kOutCols;   // weight blocks per group
  // stream-K for gate_up launches (and the 8-bit form) only: at decode sizes the
  // bf16 down's units are short (K = I), and the partial sums that end every
  // CTA's range cost more than the balance gains (measured: decode T=6
  // 96.5 -> 92.8 us, T=14 144.1 -> 142.2 us, no size slower)
  constexpr bool kStreamK = ACT == 1 || WT;

  // ---- prologue (may overlap the previous kernel of the stream): barriers,
  // tensor-map prefetch; then wait for that kernel's writes
  if (warp == 1 && lane == 0) {
    // with pairs a stage is free once both CTAs' MMAs are done with it (the
    // peer's multicast writes into this CTA's copy too)
    // (WT: an operand stage is full once every converter warp has written it)
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], WT ? kConvWarps : 1);
      mbar_init(&empty_bar[s], MC ? 2 : 1);
    }
    if (WT) {
      for (int s = 0; s < C::k8Stages; ++s) { mbar_init(&w8full_bar[s], 1); mbar_init(&w8empty_bar[s], kConvWarps); }
      for (int s = 0; s < C::kTokStages; ++s) mbar_init(&tokfull_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) { mbar_init(&tfull_bar[b], 1); mbar_init(&tempty_bar[b], 4); }
    mbar_init(done_bar, 1);
    mbar_init(table_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  } else if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_tok);
    tma_prefetch_desc(&tm_wgt);
  }
  // pairs: both CTAs' barriers exist before either multicasts into the other
  if (MC) cluster_sync_all();
  const int crank = MC ? static_cast<int>(cluster_ctarank()) : 0;
  const int wgrid = MC ? static_cast<int>(gridDim.x) / 2 : static_cast<int>(gridDim.x);   // work lists
  const int wcta = MC ? static_cast<int>(blockIdx.x) / 2 : static_cast<int>(blockIdx.x);
  // A leading phase that needs nothing from the previous kernel runs before
  // the wait on it: then the producer alone waits, builds the unit table and
  // publishes it (table_bar); otherwise every thread waits first.
  const bool pre = SWAP && !WT && args.pre_units > 0;
  const bool deferred = pre && args.pre_early != 0;
  if (!deferred) chain_wait();
  const ChainReleaseAtExit release_next;
  const int kblocks = args.K / kBK;
  // ---- unit table (warp 0): checks, unit prefix per group, split choice
  auto build_table = [&]() {
    if (deferred) {   // (otherwise every thread has loaded the offsets)
      for (int i = lane; i <= G; i += 32) s_off[i] = args.offsets ? args.offsets[i] : (i == 0 ? 0 : args.rows_max);
      __syncwarp();
    }
    const int per = (G + 31) / 32;
    const int g0 = lane * per;
    int local = 0, mx = 0;
    bool bad = false;
    for (int i = 0; i < per; ++i) {
      const int g = g0 + i;
      if (g < G) {
        const int a = s_off[g], b = s_off[g + 1];
        if (a < 0 || b < a || b > args.rows_max) bad = true;
        const int rows = bad ? 0 : b - a;
        mx = max(mx, rows);
        s_ustart[g] = local;
        // pairs: (tiles / 2) weight-sharing units per block, + NB / 2 token-sharing ones for an odd tile
        local += ((rows + C::kUnitRows - 1) / C::kUnitRows) * (MC ? NB / 2 : NB);
      }
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int base = incl - local;
    for (int i = 0; i < per; ++i)
      if (g0 + i < G) s_ustart[g0 + i] += base;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const bool any_bad = __any_sync(0xffffffffu, bad);
    const int units = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) {
      int mode = 0, S = 1, P = 1;
      if (SWAP && args.counters && mx <= kSplitRows && units > 0 && units <= args.unit_cap)
        choose_split(units, kblocks, static_cast<int>(gridDim.x), args.split_cap, kStreamK, mode, S, P);
      s_split[0] = mode;
      s_split[6] = P;
      s_split[7] = S;
      *s_total = any_bad ? 0 : units;
      if (any_bad && blockIdx.x == 0) set_status(args.status, MOE_ERR_DEVICE_CHECK);
    }
    __syncwarp();
  };
  if (!deferred) {
    // ---- group offsets into shared memory (all threads)
    for (int i = threadIdx.x; i <= G; i += kThreads)
      s_off[i] = args.offsets ? args.offsets[i] : (i == 0 ? 0 : args.rows_max);
    __syncthreads();
    if (warp == 0) build_table();
    __syncthreads();
    // a CTA without work (or every CTA, when the offsets failed their check)
    // leaves before it allocates tensor memory (with a leading phase, every CTA stays)
    if (!pre && (*s_total == 0 || WorkIter(s_split[0], s_split[7], *s_total, kblocks, wgrid, wcta).empty())) return;
  }
  // the routed phase's plan (read once the table is built) and the leading phase's (the same in every thread)
  const int units = deferred ? 0 : *s_total;
  const int mode = deferred ? 0 : s_split[0];
  const int S = deferred ? 1 : s_split[7];
  auto phase_r = [&]() { return Phase{s_split[0], s_split[7], s_split[6], *s_total, kblocks, false}; };
  int pre_mode = 0, pre_S = 1, pre_P = 1;
  const int pre_kblocks = pre ? args.pre_K / kBK : 0;
  if (pre && args.pre_counters && args.pre_rows <= kSplitRows)
    choose_split(args.pre_units, pre_kblocks, static_cast<int>(gridDim.x), args.pre_split_cap, kStreamK, pre_mode,
                 pre_S, pre_P);
  const Phase phase_s{pre_mode, pre_S, pre_P, pre ? args.pre_units : 0, pre_kblocks, true};
  // (deferred) the unit table is there once table_bar flips
  auto wait_table = [&]() { return mbar_wait(table_bar, 0, abort_flag, args.status, args.wait_ns); };
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // unit index -> group g, this CTA's first token row, token rows, weight block;
  // kind (pairs): 0 = the pair shares the weight block, 1 = the token tile
  auto decode = [&](int idx, int& g, int& row0, int& nrows, int& wb, int& kind) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {                      // last g with ustart[g] <= idx
      const int mid = (lo + hi + 1) >> 1;
      if (s_ustart[mid] <= idx) lo = mid; else hi = mid - 1;
    }
    g = lo;
    const int rows = s_off[g + 1] - s_off[g];
    const int nrb = (rows + C::kUnitRows - 1) / C::kUnitRows;
    const int local = idx - s_ustart[g];
    kind = 0;
    if (MC) {
      const int np = nrb / 2;              // tile pairs
      if (local < np * NB) {               // tiles 2rb and 2rb+1, one weight block
        const int rb = local % np;
        wb = local / np;
        row0 = s_off[g] + (2 * rb + crank) * 128;
        nrows = min(rows - (2 * rb + crank) * 128, 128);
      } else {                             // the odd last tile, weight blocks 2j and 2j+1
        kind = 1;
        wb = 2 * (local - np * NB) + crank;
        row0 = s_off[g] + (nrb - 1) * 128;
        nrows = rows - (nrb - 1) * 128;
      }
      return;
    }
    const int rb = local % nrb;
    wb = local / nrb;
    row0 = s_off[g] + rb * C::kUnitRows;
    nrows = min(rows - rb * C::kUnitRows, C::kUnitRows);
  };

  const int wrows = ACT == 1 ? 2 * args.N : args.N;   // weight rows per group
  // the leading phase: one group of pre_rows rows from row 0, weight block = unit
  auto decode_ph = [&](const Phase& ph, int idx, int& g, int& row0, int& nrows, int& wb, int& kind) {
    if (ph.pre) {
      g = 0;
      row0 = 0;
      nrows = args.pre_rows;
      wb = idx;
      kind = 0;
      return;
    }
    decode(idx, g, row0, nrows, wb, kind);
  };

  if (warp == 0 && WT) {
    // ------------------------------------------------------------ 8-bit weight producer
    // lane 0 streams the e4m3 weight tiles of each stage (gate and up, or the
    // plain rows; 128 rows x kKB * 64 codes each) into the 8-bit ring, as far
    // ahead as it goes
    const uint64_t pol_w = l2_policy_evict_first();
    long long issued = 0;
    int s8 = 0;
    uint32_t ph8 = 0;
    if (lane == 0) {
      WorkIter wi(mode, S, units, kblocks, wgrid, wcta);
      Piece pc;
      bool ok = true;
      while (ok && wi.next(pc)) {
        int g, row0, nrows, wb, kind;
        decode(pc.u, g, row0, nrows, wb, kind);
        const int wrow = g * wrows + wb * C::kOutCols;
        for (int kb = pc.kb0; kb < pc.kb1; kb += C::kKB) {
          if (!mbar_wait(&w8empty_bar[s8], ph8 ^ 1u, abort_flag, args.status, args.wait_ns)) { ok = false; break; }
          uint8_t* dst = w8_base + s8 * C::k8Bytes;
          // (a stage cut short by the piece's end still loads the whole box: the
          // codes past the piece are not used, those past K are zero-filled)
          mbar_arrive_expect_tx(&w8full_bar[s8], C::k8Bytes);
          tma_load_2d(dst, &tm_wgt, &w8full_bar[s8], kb * kBK, wrow, pol_w);
          if (ACT == 1) tma_load_2d(dst + 128 * C::k8Row, &tm_wgt, &w8full_bar[s8], kb * kBK, wrow + args.N, pol_w);
          ++issued;
          if (++s8 == C::k8Stages) { s8 = 0; ph8 ^= 1u; }
        }
      }
      // drain: every tile issued has landed before the CTA may exit
      constexpr int n8 = C::k8Stages > 0 ? C::k8Stages : 1;
      for (int s = 0; s < C::k8Stages; ++s) {
        const long long fills = issued / n8 + (s < issued % n8 ? 1 : 0);
        if (fills > 0) mbar_wait_timed(&w8full_bar[s], static_cast<uint32_t>((fills - 1) & 1), args.status);
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // lane 0 issues the copies; with gathered rows the whole warp first
    // stages the unit's source row indices in shared memory
    const uint64_t pol_tok = l2_policy_evict_last();
    const uint64_t pol_w = args.stream_w ? l2_policy_evict_first() : l2_policy_evict_normal();
    long long issued = 0;
    int stage = 0;
    uint32_t phase = 0;
    auto produce = [&](const Phase& ph) -> bool {
    WorkIter wi(ph.mode, ph.S, ph.units, ph.kblocks, wgrid, wcta);
    Piece pc;
    // the leading phase: its own operand maps and weight rows, token rows straight from the map
    const CUtensorMap* mt = ph.pre ? &tm_tok2 : &tm_tok;
    const CUtensorMap* mw = ph.pre ? &tm_wgt2 : &tm_wgt;
    const int nw = ph.pre ? args.pre_N : args.N;
    const int32_t* a_rows = ph.pre ? nullptr : args.a_rows;
    while (wi.next(pc)) {
      int g, row0, nrows, wb, kind;
      decode_ph(ph, pc.u, g, row0, nrows, wb, kind);
      const int wrow = g * (ACT == 1 ? 2 * nw : nw) + wb * C::kOutCols;
      const int n16 = (nrows + 15) >> 4;
      // token rows fetched: SWAP 16-row multiples; tokens-on-M all 128 rows
      // (whole box) or, gathered, the live rows rounded up to 4
      const int nfetch = SWAP ? n16 * 16 : (a_rows ? (nrows + 3) & ~3 : kBM_rows);
      if (a_rows) {
        __syncwarp();
        for (int i = lane; i < nfetch; i += 32) s_gidx[i] = a_rows[row0 + min(i, nrows - 1)];
        __syncwarp();
      }
      const uint32_t bytes = static_cast<uint32_t>(C::kABytes * (SWAP ? 1 : 0) + C::kBBytes * (SWAP ? 0 : 1) +
                                                   nfetch * kBK * 2);
      bool ok = true;
      if (lane == 0) {
        for (int kb = pc.kb0; kb < pc.kb1; kb += C::kKB) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, args.status, args.wait_ns)) { ok = false; break; }
          uint8_t* sa = stage_base + stage * C::kStageBytes;
          uint8_t* sb = sa + C::kKB * C::kABytes;
          const int kc = kb * kBK;
          if (SWAP) {
            // the stage's K blocks: weight tile(s) of block q at sa + q * kABytes, its token rows at
            // sb + q * (W rows x 128 bytes)
            const int nkb = pc.kb1 - kb < C::kKB ? pc.kb1 - kb : C::kKB;
            mbar_arrive_expect_tx(&full_bar[stage], nkb * bytes);
            for (int q = 0; q < nkb; ++q) {
              const int kq = kc + q * kBK;
              uint8_t* aq = sa + q * C::kABytes;
              uint8_t* bq = sb + q * (W * kBK * 2);
              tma_load_2d(aq, mw, &full_bar[stage], kq, wrow, pol_w);
              if (ACT == 1) tma_load_2d(aq + kTileRows128, mw, &full_bar[stage], kq, wrow + nw, pol_w);
              if (a_rows) {
                for (int j = 0; j < nfetch; j += 4)
                  tma_gather4(bq + j * kBK * 2, mt, &full_bar[stage], kq, s_gidx[j], s_gidx[j + 1],
                              s_gidx[j + 2], s_gidx[j + 3], pol_tok);
              } else {
                for (int j = 0; j < n16; ++j)
                  tma_load_2d(bq + j * 16 * kBK * 2, mt, &full_bar[stage], kq, row0 + 16 * j, pol_tok);
              }
            }
            ++issued;
            if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
            continue;
          }
          mbar_arrive_expect_tx(&full_bar[stage], bytes);
          uint8_t* stok = sa;   // (tokens-on-M: the token rows go first)
          if (MC) {
            // weight rows in two 128-row halves: gate | up with SiLU*mul, else rows
            // 0..127 | 128..255 of the block; a weight-sharing pair loads one half
            // per CTA, to both
            const int second = ACT == 1 ? args.N : 128;
            if (kind == 0) {
              tma_load_2d_mc(sb + crank * kTileRows128, &tm_wgt, &full_bar[stage], kc, wrow + crank * second,
                             kPairMask, pol_w);
            } else {
              tma_load_2d(sb, &tm_wgt, &full_bar[stage], kc, wrow, pol_w);
              tma_load_2d(sb + kTileRows128, &tm_wgt, &full_bar[stage], kc, wrow + second, pol_w);
            }
          } else {
            if (ACT == 1) {
              tma_load_2d(sb, &tm_wgt, &full_bar[stage], kc, wrow, pol_w);
              tma_load_2d(sb + (W / 2) * kBK * 2, &tm_wgt, &full_bar[stage], kc, wrow + args.N, pol_w);
            } else {
              tma_load_2d(sb, &tm_wgt, &full_bar[stage], kc, wrow, pol_w);
            }
          }
          if (a_rows) {
            for (int j = 0; j < nfetch; j += 4)
              tma_gather4(stok + j * kBK * 2, &tm_tok, &full_bar[stage], kc, s_gidx[j], s_gidx[j + 1],
                          s_gidx[j + 2], s_gidx[j + 3], pol_tok);
          } else if (MC) {
            // token rows in two 64-row halves; a token-sharing pair loads one half
            // per CTA, to both
            if (kind == 0) {
              tma_load_2d(stok, &tm_tok, &full_bar[stage], kc, row0, pol_tok);
              tma_load_2d(stok + kTokHalf, &tm_tok, &full_bar[stage], kc, row0 + 64, pol_tok);
            } else {
              tma_load_2d_mc(stok + crank * kTokHalf, &tm_tok, &full_bar[stage], kc, row0 + crank * 64, kPairMask,
                             pol_tok);
            }
          } else {
            const int kca = args.a_kblocks ? (kb % args.a_kblocks) * kBK : kc;
            tma_load_2d(stok, &tm_tok, &full_bar[stage], kca, row0, pol_tok);
          }
          ++issued;
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) return false;
    }
    return true;
    };
    bool run = !pre || produce(phase_s);
    if (run && deferred) {
      // the routed rows: wait for the previous kernel now, then build and publish the unit table
      chain_wait();
      build_table();
      if (lane == 0) mbar_arrive(table_bar);
    }
    if (run) produce(phase_r());
    if (lane == 0) {
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
      auto mma = [&](const Phase& ph) -> bool {
      WorkIter wi(ph.mode, ph.S, ph.units, ph.kblocks, wgrid, wcta);
      Piece pc;
      for (; wi.next(pc); ++it) {
        const int ab = C::kNumAcc == 2 ? (it & 1) : 0;
        const uint32_t aphase = (C::kNumAcc == 2 ? (it >> 1) : it) & 1;
        uint32_t idesc;
        int chains = 1, cw = 0;
        if (SWAP) {
          int g, row0, nrows, wb, kind;
          decode_ph(ph, pc.u, g, row0, nrows, wb, kind);
          const int n16 = (nrows + 15) >> 4;
          idesc = idesc_bf16_f32(128, n16 * 16);
          chains = swap_chains(n16, C::kAccCols, ACT == 1);
          cw = n16 * 16;
        } else {
          idesc = idesc_bf16_f32(128, W);
        }
        if (!mbar_wait(&tempty_bar[ab], aphase ^ 1u, abort_flag, args.status, args.wait_ns)) return false;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + ab * C::kAccCols;
        // the accumulator chains' addresses (gate or plain chains, then up chains)
        uint32_t dacc[8];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          dacc[c] = d_tmem + (c & (chains - 1)) * cw;
          dacc[4 + c] = d_tmem + (chains + (c & (chains - 1))) * cw;
        }
        const int kb0 = pc.kb0;
        bool ok = true;
        for (int kb = kb0; kb < pc.kb1; kb += C::kKB) {
          if (!mbar_wait(&full_bar[stage], phase, abort_flag, args.status, args.wait_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(stage_base + stage * C::kStageBytes);
          const uint32_t sb = WT ? smem_u32(tok_base + stage * C::kBBytes) : sa + C::kKB * C::kABytes;
          const uint64_t da = smem_desc_k128(sa);
          const uint64_t db = smem_desc_k128(sb);
          if (WT) {
            // A from tensor memory: 8 columns per 16-element K step (the up
            // tile kKB * 32 columns on); B: the stage's token tile of each K
            // block (W rows x 128 bytes, one after the other).  Every operand
            // is formed before the first MMA (the issue loop is the bound).
            const bool full_stage = pc.kb1 - kb >= C::kKB;
            const uint32_t ta0 = tmem_base + C::kAColBase + stage * C::kACols;
            uint64_t dbq[C::kKB];
#pragma unroll
            for (int q = 0; q < C::kKB; ++q) dbq[q] = smem_desc_k128(sb + q * (W * kBK * 2));
            const bool first = kb == kb0;
#pragma unroll
            for (int kk = 0; kk < C::kKB * (kBK / 16); ++kk) {
              if (kk < kBK / 16 || full_stage) {
                // (dacc[kk & 3] is chain kk & (chains - 1): chains <= 4)
                const uint32_t acc = (!first || kk >= chains) ? 1u : 0u;
                const uint64_t dbk = dbq[kk >> 2] + static_cast<uint64_t>((kk & 3) * 2);
                umma_bf16_ts(dacc[kk & 3], ta0 + kk * 8, dbk, idesc, acc);
                if (ACT == 1) umma_bf16_ts(dacc[4 + (kk & 3)], ta0 + C::kKB * kBK / 2 + kk * 8, dbk, idesc, acc);
              }
            }
          }
          if (SWAP && !WT) {
            // the stage's K blocks q: weight tile(s) at sa + q * kABytes, token rows at
            // sb + q * (W rows x 128 bytes); every operand formed before the first MMA
            const bool full_stage = pc.kb1 - kb >= C::kKB;
            uint64_t daq[C::kKB], duq[C::kKB], dbq[C::kKB];
#pragma unroll
            for (int q = 0; q < C::kKB; ++q) {
              daq[q] = smem_desc_k128(sa + q * C::kABytes);
              duq[q] = smem_desc_k128(sa + q * C::kABytes + kTileRows128);
              dbq[q] = smem_desc_k128(sb + q * (W * kBK * 2));
            }
            const bool first = kb == kb0;
#pragma unroll
            for (int kk = 0; kk < C::kKB * (kBK / 16); ++kk) {
              if (kk < kBK / 16 || full_stage) {
                // (dacc[kk & 3] is chain kk & (chains - 1): chains <= 4; +32 bytes per K step)
                const uint32_t acc = (!first || kk >= chains) ? 1u : 0u;
                const uint64_t ka = static_cast<uint64_t>((kk & 3) * 2);
                umma_bf16(dacc[kk & 3], daq[kk >> 2] + ka, dbq[kk >> 2] + ka, idesc, acc);
                if (ACT == 1) umma_bf16(dacc[4 + (kk & 3)], duq[kk >> 2] + ka, dbq[kk >> 2] + ka, idesc, acc);
              }
            }
          }
#pragma unroll
          for (int kk = 0; kk < (SWAP ? 0 : kBK / 16); ++kk) {
            // +32 bytes per 16-element K step inside the 128-byte swizzle row
            const uint64_t ka = static_cast<uint64_t>(kk * 2);
            {
              umma_bf16(d_tmem, da + ka, db + ka, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
            }
          }
          // frees the smem stage when these MMAs finish (in both CTAs of a pair)
          if (MC)
            umma_commit_mc(&empty_bar[stage], kPairMask);
          else
            umma_commit(&empty_bar[stage]);
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) return false;
        umma_commit(&tfull_bar[ab]);           // accumulator ab ready for the epilogue
      }
      return true;
      };
      if ((!pre || mma(phase_s)) && (!deferred || wait_table())) mma(phase_r());
      // every MMA issued above has completed once done_bar flips
      umma_commit(done_bar);
      mbar_wait_timed(done_bar, 0, args.status);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                    // TMEM lane quadrant of this warp
    const int lrow = q * 32 + lane;            // TMEM lane = accumulator row
    int it = 0;
    auto epilogue = [&](const Phase& ph) -> bool {
    WorkIter wi(ph.mode, ph.S, ph.units, ph.kblocks, wgrid, wcta);
    Piece pc;
    const int P = ph.P;
    // the leading phase writes its own output with its own split scratch
    __nv_bfloat16* const out = ph.pre ? args.pre_out : args.out;
    const int ldo = ph.pre ? args.pre_N : args.N;
    int* const counters = ph.pre ? args.pre_counters : args.counters;
    float* const partials = ph.pre ? args.pre_partials : args.partials;
    for (; wi.next(pc); ++it) {
      const int ab = C::kNumAcc == 2 ? (it & 1) : 0;
      const uint32_t aphase = (C::kNumAcc == 2 ? (it >> 1) : it) & 1;
      const int u = pc.u;
      int g, row0, nrows, wb, kind;
      decode_ph(ph, u, g, row0, nrows, wb, kind);
      // the warp leaves together or not at all (tcgen05.ld below is warp-wide)
      // (8-bit weights: the converter warps need the issue slots while this waits)
      bool ok = __all_sync(0xffffffffu, WT ? mbar_wait_sleep(&tfull_bar[ab], aphase, abort_flag, args.status,
                                                             args.wait_ns, 256)
                                           : mbar_wait(&tfull_bar[ab], aphase, abort_flag, args.status, args.wait_ns));
      if (P > 1) {
        // the split path meets at named barriers: the four warps leave together or not at all
        if (lane == 0) s_split[2 + q] = ok ? 1 : 0;
        epi_bar_sync();
        ok = s_split[2] && s_split[3] && s_split[4] && s_split[5];
      }
      if (!ok) return false;
      tc_fence_after();
      const uint32_t t_acc = tmem_base + ab * C::kAccCols + (static_cast<uint32_t>(q * 32) << 16);
      auto release_acc = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty_bar[ab]);
      };
      if (SWAP) {
        // accumulator row = output column wb*128 + lrow; accumulator column =
        // token, chain c of gate (h = 0) / up (h = 1) at column (h*C + c)*cw
        __nv_bfloat16* ocol = out + static_cast<size_t>(row0) * ldo + wb * 128 + lrow;
        // 8-bit weights: this accumulator row's scales (gate and up rows, or the row)
        float sg_scale = 1.f, su_scale = 1.f;
        if (WT) {
          const size_t wr0 = static_cast<size_t>(g) * wrows + wb * 128 + lrow;
          sg_scale = __ldg(args.wscale + wr0);
          if (ACT == 1) su_scale = __ldg(args.wscale + wr0 + args.N);
        }
        auto out_value = [&](float gv, float uv) {
          if (WT) { gv *= sg_scale; uv *= su_scale; }
          return ACT == 1 ? gv / (1.0f + __expf(-gv)) * uv : gv;
        };
        const int n16 = (nrows + 15) >> 4;
        const int chains = swap_chains(n16, C::kAccCols, ACT == 1);
        const int cw = n16 * 16;
        // sums of the chains for tokens [16j, 16j + 16): gs (gate or plain), us (up)
        auto load_chunk = [&](int j, float (&gs)[16], float (&us)[16]) {
#pragma unroll
          for (int i = 0; i < 16; ++i) { gs[i] = 0.f; us[i] = 0.f; }
          for (int c = 0; c < chains; ++c) {
            uint32_t r[16];
            tmem_ld_16cols(t_acc + c * cw + j * 16, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) gs[i] += __uint_as_float(r[i]);
          }
          if (ACT == 1) {
            for (int c = 0; c < chains; ++c) {
              uint32_t r[16];
              tmem_ld_16cols(t_acc + (chains + c) * cw + j * 16, r);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 16; ++i) us[i] += __uint_as_float(r[i]);
            }
          }
        };
        if (pc.np == 1) {
#pragma unroll 1
          for (int j = 0; j < n16; ++j) {
            float gs[16], us[16];
            load_chunk(j, gs, us);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              if (j * 16 + i < nrows) {
                const float h = out_value(gs[i], us[i]);
                ocol[static_cast<size_t>(j * 16 + i) * ldo] = __float2bfloat16_rn(h);
              }
            }
          }
          release_acc();
        } else {
          // a piece of a unit cut between CTAs (nrows <= 16: one 16-token
          // chunk holds the whole partial)
          constexpr int PF = partial_floats<ACT>();
          float gm[16], um[16];
          load_chunk(0, gm, um);
          release_acc();
          float4* mine = reinterpret_cast<float4*>(
              partials + ((static_cast<size_t>(u) * P + pc.pi) * 128 + lrow) * PF);
          const int n4 = (nrows + 3) >> 2;   // float4s per half that hold live tokens
#pragma unroll
          for (int i = 0; i < kSplitRows / 4; ++i) {
            if (i < n4) {
              mine[i] = make_float4(gm[4 * i], gm[4 * i + 1], gm[4 * i + 2], gm[4 * i + 3]);
              if (ACT == 1) mine[kSplitRows / 4 + i] = make_float4(um[4 * i], um[4 * i + 1], um[4 * i + 2], um[4 * i + 3]);
            }
          }
          __threadfence();
          epi_bar_sync();
          if (threadIdx.x == 64) {
            const int old = atomicAdd(&counters[u], 1);
            int last = 0;
            if (old == pc.np - 1) {
              last = 1;
              atomicExch(&counters[u], 0);   // every ticket of this unit is taken: back to zero
            } else if (old < 0 || old >= pc.np) {
              set_status(args.status, MOE_ERR_DEVICE_CHECK);   // counters were not zero at entry
            }
            s_split[1] = last;
          }
          epi_bar_sync();
          if (s_split[1]) {
            __threadfence();
            float gs[kSplitRows], us[kSplitRows];
#pragma unroll
            for (int i = 0; i < kSplitRows; ++i) { gs[i] = 0.f; us[i] = 0.f; }
            const float4* slot0 = reinterpret_cast<const float4*>(
                partials + (static_cast<size_t>(u) * P * 128 + lrow) * PF);
            const size_t slot_f4 = static_cast<size_t>(128) * PF / 4;   // float4s per piece slot
#pragma unroll
            for (int i = 0; i < kSplitRows / 4; ++i) {
              if (i >= n4) break;
              // pieces in order, whoever arrived last; the loads of all pieces
              // are independent and go out together
#pragma unroll 8
              for (int j = 0; j < pc.np; ++j) {
                float4 a, b;
                if (j == pc.pi) {
                  a = make_float4(gm[4 * i], gm[4 * i + 1], gm[4 * i + 2], gm[4 * i + 3]);
                  b = make_float4(um[4 * i], um[4 * i + 1], um[4 * i + 2], um[4 * i + 3]);
                } else {
                  a = __ldcg(slot0 + j * slot_f4 + i);
                  b = ACT == 1 ? __ldcg(slot0 + j * slot_f4 + kSplitRows / 4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                gs[4 * i] += a.x; gs[4 * i + 1] += a.y; gs[4 * i + 2] += a.z; gs[4 * i + 3] += a.w;
                us[4 * i] += b.x; us[4 * i + 1] += b.y; us[4 * i + 2] += b.z; us[4 * i + 3] += b.w;
              }
            }
#pragma unroll
            for (int i = 0; i < kSplitRows; ++i) {
              if (i < nrows) {
                const float h = out_value(gs[i], us[i]);
                ocol[static_cast<size_t>(i) * ldo] = __float2bfloat16_rn(h);
              }
            }
          }
        }
      } else {
        // accumulator row = token row0 + lrow; accumulator column = output column
        const bool live = lrow < nrows;
        __nv_bfloat16* orow = args.out + static_cast<size_t>(row0 + lrow) * args.N + wb * C::kOutCols;
        if (ACT == 2) {
          // fp32 output, no rounding (router logits)
          float* orow32 = reinterpret_cast<float*>(args.out) + static_cast<size_t>(row0 + lrow) * args.N +
                          wb * C::kOutCols;
#pragma unroll 1
          for (int c = 0; c < W; c += 32) {
            uint32_t r[32];
            tmem_ld_32cols(t_acc + c, r);
            tmem_ld_wait();
            if (live) {
              float4* dst = reinterpret_cast<float4*>(orow32 + c);
#pragma unroll
              for (int v = 0; v < 8; ++v)
                dst[v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                     __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
            }
          }
        } else if (ACT == 1) {
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
        release_acc();
      }
    }
    return true;
    };
    if ((!pre || epilogue(phase_s)) && (!deferred || wait_table())) epilogue(phase_r());
  } else if (WT && warp == 6 + kConvWarps) {
    // ------------------------------------------------------------ token producer
    // lane 0 loads the token tile of each K block (the unit's rows: 16-row
    // tiles, or gathered rows) into the token ring; with gathered rows the
    // whole warp first stages the unit's source rows
    const uint64_t pol_tok = l2_policy_evict_last();
    long long issued = 0;
    int st = 0;
    uint32_t pht = 0;
    WorkIter wi(mode, S, units, kblocks, wgrid, wcta);
    Piece pc;
    while (wi.next(pc)) {
      int g, row0, nrows, wb, kind;
      decode(pc.u, g, row0, nrows, wb, kind);
      const int n16 = (nrows + 15) >> 4;
      const int nfetch = n16 * 16;
      if (args.a_rows) {
        __syncwarp();
        for (int i = lane; i < nfetch; i += 32) s_gidx[i] = args.a_rows[row0 + min(i, nrows - 1)];
        __syncwarp();
      }
      bool ok = true;
      if (lane == 0) {
        for (int kb = pc.kb0; kb < pc.kb1; kb += C::kKB) {
          const int nkb = pc.kb1 - kb < C::kKB ? pc.kb1 - kb : C::kKB;
          // the slot is free once the MMAs of its A stage's previous use are done
          if (!mbar_wait(&empty_bar[st], pht ^ 1u, abort_flag, args.status, args.wait_ns)) { ok = false; break; }
          mbar_arrive_expect_tx(&tokfull_bar[st], static_cast<uint32_t>(nkb * nfetch * kBK * 2));
          for (int q = 0; q < nkb; ++q) {
            const int kc = (kb + q) * kBK;
            uint8_t* stok = tok_base + st * C::kBBytes + q * (W * kBK * 2);
            if (args.a_rows) {
              for (int j = 0; j < nfetch; j += 4)
                tma_gather4(stok + j * kBK * 2, &tm_tok, &tokfull_bar[st], kc, s_gidx[j], s_gidx[j + 1],
                            s_gidx[j + 2], s_gidx[j + 3], pol_tok);
            } else {
              for (int j = 0; j < n16; ++j)
                tma_load_2d(stok + j * 16 * kBK * 2, &tm_tok, &tokfull_bar[st], kc, row0 + 16 * j, pol_tok);
            }
          }
          ++issued;
          if (++st == C::kTokStages) { st = 0; pht ^= 1u; }
        }
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
    }
    if (lane == 0) {
      // drain: every tile issued has landed before the CTA may exit
      constexpr int nt = C::kTokStages > 0 ? C::kTokStages : 1;
      for (int s = 0; s < C::kTokStages; ++s) {
        const long long fills = issued / nt + (s < issued % nt ? 1 : 0);
        if (fills > 0) mbar_wait_timed(&tokfull_bar[s], static_cast<uint32_t>((fills - 1) & 1), args.status);
      }
    }
  } else if constexpr (WT) {
    // ------------------------------------------------------------ converters
    // warps 6..13: an 8-bit weight stage -> bf16 A stage in tensor memory.  A
    // warp may touch only its lane quadrant (warp mod 4), so each thread owns
    // one weight row r of the tile: with gate and up tiles the quadrant's first
    // warp widens the gate row and its second the up row (64 codes -> 32
    // columns per K block); a plain tile is split in K halves (32 codes -> 16
    // columns per K block).  The 8-bit tile comes in the 128-byte swizzle, in
    // which the 16-byte chunk c of row r sits at chunk c ^ (r & 7), so that the
    // row-per-lane reads meet no bank conflicts.  A stage is full when every
    // converter warp's stores have completed and its token tiles have landed.
    const int quad = warp & 3;
    const int half = (warp - 6) >> 2;
    const int r = quad * 32 + lane;
    const uint32_t rsw = static_cast<uint32_t>(r & 7);
    const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + C::kAColBase;
    int stage = 0, s8 = 0;
    uint32_t phase = 0, ph8 = 0;
    bool ok = true;
    WorkIter wi(mode, S, units, kblocks, wgrid, wcta);
    Piece pc;
    while (ok && wi.next(pc)) {
      for (int kb = pc.kb0; kb < pc.kb1; kb += C::kKB) {
       const int nkb = pc.kb1 - kb < C::kKB ? pc.kb1 - kb : C::kKB;
       ok = __all_sync(0xffffffffu, mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, args.status, args.wait_ns));
       if (!ok) break;
       tc_fence_after();
       ok = __all_sync(0xffffffffu, mbar_wait(&w8full_bar[s8], ph8, abort_flag, args.status, args.wait_ns));
       if (!ok) break;
       const uint32_t row8 = smem_u32(w8_base + s8 * C::k8Bytes) + (ACT == 1 ? half * 128 * C::k8Row : 0) + r * C::k8Row;
       // the stage's K blocks: chunks 4q .. 4q + 3 of the row
       for (int q = 0; q < nkb; ++q) {
        // gate / up rows: K block q at column q * 32 of the tile's kKB * 32;
        // plain rows: K block q at column q * 32, this warp's K half 16 on
        const uint32_t dst = t_row + stage * C::kACols + q * (kBK / 2);
        if (ACT == 1) {
          uint4 v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) v[j] = lds_u4(row8 + ((static_cast<uint32_t>(4 * q + j) ^ rsw) << 4));
          uint32_t o[32];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint2 a0 = e4m3x4_to_bf16x4(v[j].x), a1 = e4m3x4_to_bf16x4(v[j].y);
            const uint2 a2 = e4m3x4_to_bf16x4(v[j].z), a3 = e4m3x4_to_bf16x4(v[j].w);
            o[8 * j + 0] = a0.x; o[8 * j + 1] = a0.y; o[8 * j + 2] = a1.x; o[8 * j + 3] = a1.y;
            o[8 * j + 4] = a2.x; o[8 * j + 5] = a2.y; o[8 * j + 6] = a3.x; o[8 * j + 7] = a3.y;
          }
          tmem_st_32cols(dst + half * (C::kKB * kBK / 2), o);
        } else {
          uint4 v[2];
#pragma unroll
          for (int j = 0; j < 2; ++j) v[j] = lds_u4(row8 + ((static_cast<uint32_t>(4 * q + 2 * half + j) ^ rsw) << 4));
          uint32_t o[16];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint2 a0 = e4m3x4_to_bf16x4(v[j].x), a1 = e4m3x4_to_bf16x4(v[j].y);
            const uint2 a2 = e4m3x4_to_bf16x4(v[j].z), a3 = e4m3x4_to_bf16x4(v[j].w);
            o[8 * j + 0] = a0.x; o[8 * j + 1] = a0.y; o[8 * j + 2] = a1.x; o[8 * j + 3] = a1.y;
            o[8 * j + 4] = a2.x; o[8 * j + 5] = a2.y; o[8 * j + 6] = a3.x; o[8 * j + 7] = a3.y;
          }
          tmem_st_16cols(dst + half * (kBK / 4), o);
        }
       }
       tmem_st_wait();
       __syncwarp();
       if (lane == 0) mbar_arrive(&w8empty_bar[s8]);   // (its codes have been read and stored)
       if (++s8 == C::k8Stages) { s8 = 0; ph8 ^= 1u; }
       // the stage is full once its token tiles have landed too
       ok = __all_sync(0xffffffffu, mbar_wait(&tokfull_bar[stage], phase, abort_flag, args.status, args.wait_ns));
       if (!ok) break;
       tc_fence_before();
       __syncwarp();
       if (lane == 0) mbar_arrive(&full_bar[stage]);
       if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
  // pairs: neither CTA leaves while the other may still arrive on its barriers
  if (MC) cluster_sync_all();
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

// 2-D byte tensor [rows][cols] (e4m3 weights), box [box_rows][128 bytes], in
// the 128-byte swizzle (the converter warps read it one row per lane).
bool make_map_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(2 * kBK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Split-K scratch of one weights-on-M launch: a ticket counter per unit and
// fp32 partial slots (at most kMaxSlots sub-units).
struct SplitPlan {
  int unit_cap = 0;
  int split_cap = 0;
  size_t partial_bytes = 0;   // 0: the launch never splits
};

constexpr int kSwapRows = 64;   // token rows per unit in the weights-on-M form
constexpr int kMaxSlots = 4096;
// Ticket counters: a fixed region at the start of every split-K scratch, the
// same size whatever the shape, so that calls of different shapes can share a
// scratch in turn (no call's partial sums ever land where another call keeps
// its counters).  Units beyond it are never split.
constexpr int kCounterInts = 16384;

SplitPlan split_plan(int G, int rows_max, int N, int act, int max_slots = kMaxSlots) {
  SplitPlan p;
  if (rows_max <= 0 || N % 128 || static_cast<long long>(rows_max) > 64LL * G) return p;
  const long long nonempty = G < rows_max ? G : rows_max;
  long long units = ((rows_max + kSwapRows - 1) / kSwapRows + nonempty) * (N / 128);
  if (units > kCounterInts) units = kCounterInts;
  const long long cap = units * kMaxSplit < max_slots ? units * kMaxSplit : max_slots;
  p.unit_cap = static_cast<int>(units);
  p.split_cap = static_cast<int>(cap);
  const size_t slot = 128 * static_cast<size_t>(act ? partial_floats<1>() : partial_floats<0>()) * sizeof(float);
  p.partial_bytes = static_cast<size_t>(cap) * slot;
  return p;
}

template <int SWAP, int W, int ACT, int MC = 0, int WT = 0>
int launch_cfg(const void* a, const void* w, const int32_t* offsets, int G, int rows_max, int N, int K, void* out,
               int* status, const GemmScratch* scratch, int grid_cap, cudaStream_t stream, int* launches,
               int max_slots = kMaxSlots, int K_a = 0, const int32_t* a_rows = nullptr, int a_src_rows = 0,
               const float* w_scale = nullptr, const LeadPhase* lead = nullptr) {
  using C = Cfg<SWAP, W, ACT, MC, WT>;
  constexpr int kThreads = C::kThreads;
  auto kernel = grouped_gemm_kernel<SWAP, W, ACT, MC, WT>;
  // per device: the shared-memory attribute set once, the pairs that fit at once
  static bool attr_done[64] = {};
  static int max_clusters[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  std::unique_lock<std::mutex> lk(mu);
  if (dev >= 64 || !attr_done[dev]) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
      return MOE_ERR_CUDA;
    int clusters = 0;
    if (MC) {
      // pairs of CTAs fit only where two SMs of one GPC are free: ask how many
      cudaLaunchConfig_t q = {};
      q.gridDim = dim3(2 * grid_cap);
      q.blockDim = dim3(kThreads);
      q.dynamicSmemBytes = C::kSmemBytes;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 2;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      q.attrs = at;
      q.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &q) != cudaSuccess || clusters < 1) return MOE_ERR_CUDA;
    }
    if (dev < 64) {
      max_clusters[dev] = clusters;
      attr_done[dev] = true;
    }
  }
  const int mc = dev < 64 ? max_clusters[dev] : 1;
  lk.unlock();
  CUtensorMap tt, tw;
  const int wrows = ACT == 1 ? 2 * N : N;
  const uint32_t tok_box = SWAP ? 16 : (MC ? 64 : 128);
  const uint32_t wgt_box = SWAP ? 128 : (ACT == 1 || MC ? W / 2 : W);
  if (a_rows) {   // rows fetched one at a time by gather4: a one-row box over the source rows
    if (!make_map(&tt, a, static_cast<uint64_t>(a_src_rows), static_cast<uint64_t>(K), 1)) return MOE_ERR_CUDA;
  } else if (!make_map(&tt, a, static_cast<uint64_t>(rows_max), static_cast<uint64_t>(K_a ? K_a : K), tok_box)) {
    return MOE_ERR_CUDA;
  }
  if (WT ? !make_map_u8(&tw, w, static_cast<uint64_t>(G) * wrows, static_cast<uint64_t>(K), wgt_box)
         : !make_map(&tw, w, static_cast<uint64_t>(G) * wrows, static_cast<uint64_t>(K), wgt_box))
    return MOE_ERR_CUDA;
  // upper bound on the unit count: every non-empty group adds at most one partial row block
  const long long nonempty = offsets ? (G < rows_max ? G : rows_max) : 1;
  long long bound = (static_cast<long long>((rows_max + C::kUnitRows - 1) / C::kUnitRows) + nonempty) *
                    (N / C::kOutCols / (MC ? 2 : 1));
  GemmArgs args{offsets, G, rows_max, N, K, reinterpret_cast<__nv_bfloat16*>(out), status, SWAP ? 1 : 0,
                nullptr, nullptr, 0, 0, K_a ? K_a / kBK : 0, a_rows, wait_limit_ns(), w_scale,
                0, 0, 0, 0, 0, nullptr, nullptr, nullptr, 0};
  // the leading phase's operand maps (without one, the launch's own maps stand in)
  CUtensorMap tt2 = tt, tw2 = tw;
  if (lead) {
    if (!SWAP || WT || !lead_phase_applies(lead->rows, lead->N, lead->K)) return MOE_ERR_UNSUPPORTED;
    const int lrows = ACT == 1 ? 2 * lead->N : lead->N;
    if (!make_map(&tt2, lead->a, static_cast<uint64_t>(lead->rows), static_cast<uint64_t>(lead->K), 16) ||
        !make_map(&tw2, lead->w, static_cast<uint64_t>(lrows), static_cast<uint64_t>(lead->K), 128))
      return MOE_ERR_CUDA;
    args.pre_units = lead->N / 128;
    args.pre_N = lead->N;
    args.pre_K = lead->K;
    args.pre_rows = lead->rows;
    args.pre_early = lead->early ? 1 : 0;
    args.pre_out = static_cast<__nv_bfloat16*>(lead->out);
    const SplitPlan lp = split_plan(1, lead->rows, lead->N, ACT, max_slots);
    if (lead->scratch.counters && lead->scratch.partials && lp.partial_bytes &&
        lead->scratch.partial_bytes >= lp.partial_bytes && args.pre_units <= lp.unit_cap) {
      args.pre_counters = lead->scratch.counters;
      args.pre_partials = static_cast<float*>(lead->scratch.partials);
      args.pre_split_cap = lp.split_cap;
    }
  }
  if (SWAP && scratch && scratch->counters && scratch->partials) {
    const SplitPlan p = split_plan(G, rows_max, N, ACT, max_slots);
    if (p.partial_bytes && scratch->partial_bytes >= p.partial_bytes) {
      args.counters = scratch->counters;
      args.partials = static_cast<float*>(scratch->partials);
      args.unit_cap = p.unit_cap;
      args.split_cap = p.split_cap;
      bound *= kMaxSplit;
    }
  }
  if (MC) {
    // one work list per pair: at most grid_cap / 2 pairs, and no more than fit at once
    long long pairs = grid_cap / 2;
    if (pairs > mc) pairs = mc;
    if (pairs > bound) pairs = bound;
    if (pairs < 1) pairs = 1;
    if (launch_chained_cluster(kernel, dim3(static_cast<int>(2 * pairs)), dim3(kThreads), C::kSmemBytes, stream, 2,
                               tt, tw, tt2, tw2, args) != cudaSuccess)
      return MOE_ERR_CUDA;
    ++*launches;
    return MOE_OK;
  }
  // (a leading phase spreads over every CTA the launch may have)
  int grid = static_cast<int>(bound < grid_cap && !lead ? bound : grid_cap);
  if (grid < 1) grid = 1;
  if (launch_chained(kernel, dim3(grid), dim3(kThreads), C::kSmemBytes, stream, tt, tw, tt2, tw2, args) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  ++*launches;
  return MOE_OK;
}

// Tokens-on-M launches with an even number of 256-wide weight blocks run as
// multicast pairs.
constexpr bool kPairs = true;

}  // namespace

bool grouped_gemm_weights_on_m(int G, int rows_max, int N) {
  return N % 128 == 0 && static_cast<long long>(rows_max) <= 64LL * G;
}

bool lead_phase_applies(int rows, int N, int K) {
  return rows >= 1 && rows <= kSplitRows && N % 128 == 0 && K % kBK == 0 && K > 0;
}

size_t grouped_gemm_counter_region_bytes() { return static_cast<size_t>(kCounterInts) * sizeof(int); }

size_t grouped_gemm_partial_bytes(int G, int rows_max, int N, int act, int max_slots) {
  return split_plan(G, rows_max, N, act, max_slots > 0 ? max_slots : kMaxSlots).partial_bytes;
}

size_t grouped_gemm_counters_used_bytes(int G, int rows_max, int N, int act) {
  return align_up(static_cast<size_t>(split_plan(G, rows_max, N, act).unit_cap) * sizeof(int));
}

size_t grouped_gemm_ws_bytes(int G, int rows_max, int N, int act, int max_slots) {
  const size_t pb = grouped_gemm_partial_bytes(G, rows_max, N, act, max_slots);
  return pb ? grouped_gemm_counter_region_bytes() + pb : 0;
}

GemmScratch grouped_gemm_scratch(void* ws, size_t ws_bytes) {
  GemmScratch s{};
  const size_t c = grouped_gemm_counter_region_bytes();
  if (ws && ws_bytes > c) {
    s.counters = static_cast<int*>(ws);
    s.partials = static_cast<uint8_t*>(ws) + c;
    s.partial_bytes = ws_bytes - c;
  }
  return s;
}

int grouped_gemm_launch(const void* a, const void* w, const int32_t* offsets, int G, int rows_max, int N, int K,
                        int act, void* out, int* status, const GemmScratch* scratch, int grid_cap, cudaStream_t stream,
                        int* launches, const int32_t* a_rows, int a_src_rows, int max_slots, int max_group_rows,
                        const float* w_scale, const LeadPhase* lead) {
  if (rows_max == 0) return MOE_OK;
  if (max_slots <= 0) max_slots = kMaxSlots;
  // groups of one row: a weight stream on the CUDA cores
  const int bound = rows_max == 1 ? 1 : max_group_rows;
  if (lead && (w_scale || act == 2)) return MOE_ERR_UNSUPPORTED;
  if (!lead && act != 2 && grouped_gemv_applies(G, N, K, act, bound))
    return grouped_gemv_launch(a, w, w_scale, offsets, G, rows_max, N, K, act, out, status, stream, launches, a_rows,
                               a_src_rows, bound, grid_cap);
  if (w_scale) {
    // 8-bit weights: the weights-on-M form only (decode-sized batches)
    if (!grouped_gemm_weights_on_m(G, rows_max, N) || act == 2) return MOE_ERR_UNSUPPORTED;
    if (act == 1)
      return launch_cfg<1, kSwapRows, 1, 0, 1>(a, w, offsets, G, rows_max, N, K, out, status, scratch, grid_cap,
                                               stream, launches, max_slots, 0, a_rows, a_src_rows, w_scale);
    return launch_cfg<1, kSwapRows, 0, 0, 1>(a, w, offsets, G, rows_max, N, K, out, status, scratch, grid_cap, stream,
                                             launches, max_slots, 0, a_rows, a_src_rows, w_scale);
  }
  if (grouped_gemm_weights_on_m(G, rows_max, N)) {
    if (act == 1)
      return launch_cfg<1, kSwapRows, 1>(a, w, offsets, G, rows_max, N, K, out, status, scratch, grid_cap, stream,
                                         launches, max_slots, 0, a_rows, a_src_rows, nullptr, lead);
    return launch_cfg<1, kSwapRows, 0>(a, w, offsets, G, rows_max, N, K, out, status, scratch, grid_cap, stream,
                                       launches, max_slots, 0, a_rows, a_src_rows, nullptr, lead);
  }
  if (lead) return MOE_ERR_UNSUPPORTED;   // (a leading phase joins weights-on-M launches of bf16 weights only)
  // the pairs multicast operand tiles inside a cluster of this GPU: only for
  // operands in this GPU's own device memory
  const bool pairs_ok = kPairs && !a_rows && grid_cap >= 2 && (N % 256 == 0 || N % 512 == 0);
  if (pairs_ok && (!device_local(a) || !device_local(w))) return MOE_ERR_UNSUPPORTED;
  if (act == 1) {
    if (N % 256 == 0 && kPairs && !a_rows && grid_cap >= 2)
      return launch_cfg<0, 256, 1, 1>(a, w, offsets, G, rows_max, N, K, out, status, nullptr, grid_cap, stream,
                                      launches);
    if (N % 128 == 0)
      return launch_cfg<0, 256, 1>(a, w, offsets, G, rows_max, N, K, out, status, nullptr, grid_cap, stream,
                                   launches, kMaxSlots, 0, a_rows, a_src_rows);
    return launch_cfg<0, 128, 1>(a, w, offsets, G, rows_max, N, K, out, status, nullptr, grid_cap, stream, launches,
                                 kMaxSlots, 0, a_rows, a_src_rows);
  }
  if (N % 512 == 0 && kPairs && !a_rows && grid_cap >= 2)
    return launch_cfg<0, 256, 0, 1>(a, w, offsets, G, rows_max, N, K, out, status, nullptr, grid_cap, stream,
                                    launches);
  if (N % 256 == 0)
    return launch_cfg<0, 256, 0>(a, w, offsets, G, rows_max, N, K, out, status, nullptr, grid_cap, stream, launches,
                                 kMaxSlots, 0, a_rows, a_src_rows);
  if (N % 128 == 0)
    return launch_cfg<0, 128, 0>(a, w, offsets, G, rows_max, N, K, out, status, nullptr, grid_cap, stream, launches,
                                 kMaxSlots, 0, a_rows, a_src_rows);
  return launch_cfg<0, 64, 0>(a, w, offsets, G, rows_max, N, K, out, status, nullptr, grid_cap, stream, launches,
                              kMaxSlots, 0, a_rows, a_src_rows);
}

int router_gemm_launch(const void* x, const void* wr3, int T, int H, int E, float* logits, int* status, int grid_cap,
                       cudaStream_t stream, int* launches) {
  if (T == 0) return MOE_OK;
  const int K = 3 * H;
  // the logits block width whose longest CTA streams the fewest bytes: rounds
  // of units per CTA x (token tile + weight block) per K block
  const long long mtiles = (T + 127) / 128;
  int best_bn = 64;
  long long best = -1;
  for (int bn = 256; bn >= 64; bn /= 2) {
    if (E % bn) continue;
    const long long units = mtiles * (E / bn);
    const long long cost = (units + grid_cap - 1) / grid_cap * (kTileRows128 + bn * kBK * 2);
    if (best < 0 || cost < best) { best = cost; best_bn = bn; }
  }
  if (best_bn == 256)
    return launch_cfg<0, 256, 2>(x, wr3, nullptr, 1, T, E, K, logits, status, nullptr, grid_cap, stream, launches,
                                 kMaxSlots, H);
  if (best_bn == 128)
    return launch_cfg<0, 128, 2>(x, wr3, nullptr, 1, T, E, K, logits, status, nullptr, grid_cap, stream, launches,
                                 kMaxSlots, H);
  return launch_cfg<0, 64, 2>(x, wr3, nullptr, 1, T, E, K, logits, status, nullptr, grid_cap, stream, launches,
                              kMaxSlots, H);
}

int grouped_gemm_max_groups() { return kMaxGroups; }

}  // namespace moe
