// Steps a4-a5 in bf16 on the 5th-generation tensor cores: the grouped expert
// GEMMs of the sparse-MoE layer ("The Evolving Transformer - 05 Mixtral",
// section 04 SwiGLU: each expert is down(silu(gate x) * up x) with three
// bias-free matrices; section 05: each expert sees only the tokens routed to
// it, and the page notes production stacks batch those tokens per expert).
//
// One persistent kernel per GEMM, one CTA per SM, warp-specialised:
//   warp 0      TMA producer: 128x64 A tile + two 128x64 B tiles per stage
//               (128-byte swizzle) into a 4-stage shared-memory ring.
//   warp 1      owns tensor memory (512 columns) and issues tcgen05.mma
//               (M=128, N=256, K=16, bf16 in, fp32 accumulate) into one of
//               two 256-column accumulators.
//   warps 2-5   epilogue: tcgen05.ld of the accumulator rows, fp32 math,
//               bf16 rounding, stores of the rows that belong to the expert
//               (large batches: 32 x 32 blocks staged through shared memory,
//               so that each store instruction writes whole row segments).
// Output tiles are 128 rows of one expert's segment x (gate/up) 128 columns
// of h, whose accumulator holds the W1 half in columns 0-127 and the W3 half
// in 128-255, or (down) 256 columns of y.  Tiles are numbered expert by
// expert, row block fastest, so CTAs running at the same time share the
// weight tile through L2.  Experts with no rows have no tiles, so their
// weights are never read.  The expert boundaries come from the device-side
// offsets[E+1]; the host never reads the per-expert counts.
//
// int8 weights (KerasFormers Mixtral docs, "Lower memory": weight-only int8,
// one fp32 scale per output row) run here in the small-batch form below;
// more rows go to ffn_w8_wide.cu.  The epilogue multiplies each accumulator
// row by its scale s[e, n] before the SwiGLU (gate/up) or the rounding
// (down): the scale of an output row factors out of its dot product.
//
// Small batches (decode).  With a few tokens per expert a 128-row token tile
// is mostly padding, and the per-stage token tile costs as much shared
// memory as the weights.  So for small row counts the roles swap: a tile is
// 256 weight rows x 32 tokens, computed as two M=128, N=32 MMAs per K step
// (weights as the A operand, the token rows as B).  The accumulator lanes are
// then weight rows: each epilogue thread owns one output column (one row
// scale) for up to 32 tokens.  A stage is the 4 KB token tile + the weights,
// so more stages fit and more weight bytes are in flight per SM.  With int8
// weights the converters write the widened weight rows straight into tensor
// memory (tcgen05.st, one row per lane, two bf16 per column) and the MMA
// takes its A operand from there: the widened weights never touch shared
// memory, whose bandwidth would otherwise bound the small-batch int8 GEMM.
// The converters are two groups of four warps taking alternate K steps: a
// group's step is a chain of shared-memory loads, widening, tensor-memory
// stores and their wait, and two groups overlap those chains.  At N=32 one
// thread issues an MMA every ~48 cycles whatever it feeds, four times the
// tensor pipe's time for it, so the int8 form issues from two threads, one
// per 128-row half (its own accumulator): 16 MMAs per 128-K stage would
// otherwise take longer to issue than the stage takes to stream.
//
// Every wait is bounded (globaltimer + iteration cap).  A wait that runs out
// raises a CTA-wide abort flag and records MOE_ETIMEOUT; each role then
// leaves its loop, the TMA issuers wait (bounded) for their copies in
// flight, the MMA warp waits (bounded) for its MMAs, and TMEM is freed
// before returning.
//
// The set-up (barriers, tensor-map prefetch, TMEM allocation) runs before the
// kernel waits on its predecessor (programmatic dependent launch), so it
// overlaps the previous kernel's tail.
#include <cuda.h>
#include <mutex>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "widen.cuh"

namespace moe {
namespace {

constexpr int BM = 128;                  // rows (tokens) per tile
constexpr int TN = 32;                   // swapped mode: tokens per tile (the MMA N)
constexpr int BK = 64;                   // K per stage: one 128-byte swizzle row of bf16
constexpr int BN_HALF = 128;             // rows of one B box
constexpr int BN = 2 * BN_HALF;          // MMA N
constexpr int UMMA_K = 16;               // K of one tcgen05.mma (bf16)
constexpr int B_HALF_BYTES = BN_HALF * BK * 2;
constexpr int EPI_THREADS = 128;
#ifndef MOE_SWAP_STAGES
#define MOE_SWAP_STAGES 6
#endif
#ifndef MOE_W8_SWAP_STAGES
#define MOE_W8_SWAP_STAGES 6
#endif
#ifndef MOE_TOK_STAGES
#define MOE_TOK_STAGES 3
#endif
#ifndef MOE_TMEM_A_STAGES
#define MOE_TMEM_A_STAGES 3
#endif
#ifndef MOE_SWAP_MAX_ROWS
#define MOE_SWAP_MAX_ROWS 128
#endif
#ifndef MOE_PREFETCH_ROW_BYTES
#define MOE_PREFETCH_ROW_BYTES 2048
#endif
constexpr int CONV_WARPS = 4;     // int8: converter warps per group, one per tensor-memory lane quarter
constexpr int CONV_GROUPS = 2;    // int8: converter groups, taking alternate K steps
constexpr int MAX_STAGES = 10;
// int8 small-batch mode: a stage covers 128 K of each weight row (128-byte
// rows in every TMA request); its widened weights sit in tensor memory as two
// 128-row halves x 128 K = 2 x 64 columns, after the 128 accumulator columns.
constexpr int BK_W = 128;
constexpr int RAW_W_HALF_BYTES = BN_HALF * BK_W;      // one 128x128 int8 box, 16 KB
constexpr int TMEM_A_STAGES = MOE_TMEM_A_STAGES;
constexpr int TMEM_A_COL0 = 128;
constexpr int TMEM_A_HALF_COLS = BK_W / 2;
constexpr int TMEM_A_STAGE_COLS = 2 * TMEM_A_HALF_COLS;
constexpr int MAX_E = 64;
constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, BN);
constexpr uint32_t IDESC_SWAP = ptx::idesc_bf16_f32(BN_HALF, TN);
// The swapped mode serves GEMMs of at most this many rows (tokens x k).
constexpr int SWAP_MAX_ROWS = MOE_SWAP_MAX_ROWS;

struct SmemCtl {
  uint64_t full[MAX_STAGES];       // a stage's TMA copies landed
  uint64_t empty[MAX_STAGES];      // the MMA (and, int8 path, every converter) is done with a stage
  uint64_t c_full[TMEM_A_STAGES];  // int8: widened weights written to tensor memory
  uint64_t c_empty[TMEM_A_STAGES]; // int8: the MMA is done with them
  uint64_t tok_full[8];            // int8 small-batch mode: token tile landed
  uint64_t tok_empty[8];           // int8 small-batch mode: the MMA is done with a token tile
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int tile_prefix[MAX_E + 1];
  int mtiles[MAX_E];
  int seg[MAX_E + 1];
};

// Plan of each mode.  A shared-memory stage is the token tile (128 rows, or
// 32 when swapped) + the bf16 weights: 4 stages (6 swapped).  int8 (always
// swapped): the weights no longer wait for the MMA (it reads them from
// tensor memory), so they get a ring of their own, 6 stages of 256 rows x
// 128 K, freed by the converters; the token tiles have a 3-stage ring with
// a producer warp of their own, freed by the MMA; 3 stages of widened
// weights in tensor memory.
template <bool W8, bool SWAP>
struct Plan {
  static_assert(!W8 || SWAP, "int8 weights: small-batch form only");
  static constexpr bool tmem_a = W8;                     // A operand (widened weights) in tensor memory
  static constexpr int kstep = tmem_a ? BK_W : BK;       // K per stage
  static constexpr int rows = SWAP ? TN : BM;            // token rows per tile
  static constexpr int tok_box_bytes = rows * BK * 2;    // one 64-wide token box
  static constexpr int a_bytes = (kstep / BK) * tok_box_bytes;  // token tile per stage
  static constexpr int b_off = tmem_a ? 0 : a_bytes;     // weights' offset in a stage
  static constexpr int stage_bytes = b_off + (W8 ? 2 * RAW_W_HALF_BYTES : 2 * B_HALF_BYTES);
  static constexpr int tok_stages = tmem_a ? MOE_TOK_STAGES : 0;  // separate token ring
  static constexpr int conv_warps = W8 ? CONV_WARPS * CONV_GROUPS : 0;  // from warp 6
  static constexpr int tok_warp = 6 + conv_warps;        // the token ring's producer (int8)
  static constexpr int issuers = tmem_a ? 2 : 1;         // MMA-issuing threads, one per 128-row half
  static constexpr int mma2_warp = tok_warp + 1;         // the second issuer's warp (int8)
  static constexpr int stages = SWAP ? (W8 ? MOE_W8_SWAP_STAGES : MOE_SWAP_STAGES) : 4;
  static constexpr int threads = 192 + 32 * conv_warps + (tmem_a ? 64 : 0);
  static constexpr int acc_cols = SWAP ? 2 * TN : BN;    // fp32 columns of one accumulator
  static constexpr int tmem_cols = (SWAP && !W8) ? 128 : 512;  // power of two
  static_assert(!tmem_a || TMEM_A_COL0 + TMEM_A_STAGES * TMEM_A_STAGE_COLS <= 512, "tensor-memory ring too deep");
  static_assert(!tmem_a || 2 * acc_cols <= TMEM_A_COL0, "accumulators overlap the widened weights");
  static_assert(tok_stages <= 8, "token ring too deep");
  static constexpr size_t ring_bytes = static_cast<size_t>(stages) * stage_bytes +
                                       static_cast<size_t>(tok_stages) * a_bytes;
  static constexpr size_t ctl_bytes = (sizeof(SmemCtl) + 127) / 128 * 128;
  // Large-batch mode: one 32 x 64-byte staging block per epilogue warp.
  static constexpr size_t stg_bytes = SWAP ? 0 : 4 * 32 * 64;
  static constexpr size_t smem_bytes = 1024 + ring_bytes + ctl_bytes + stg_bytes;
  static_assert(stages <= MAX_STAGES, "too many stages");
  static_assert(smem_bytes <= 227 * 1024, "plan exceeds shared memory");
  static_assert(2 * acc_cols <= tmem_cols, "accumulators exceed the tensor-memory allocation");
};

struct GemmArgs {
  const int32_t* offsets;  // [E+1], device
  const uint8_t* b0;       // the weights B0, B1 (B1 null for down), rows of K elements
  const uint8_t* b1;
  int b_esz;               // bytes per weight element
  __nv_bfloat16* out;      // [Tk, ldo]
  const float* scale0;     // int8 path: row scales of B0 [E * b_rows]
  const float* scale1;     // int8 path: row scales of B1 (gate/up only)
  __nv_bfloat16* keep;     // bf16 gate/up, optional (training): the SwiGLU's
                           // local derivatives, planes [2, Tk, ldo] (see keep_pair)
  int ldo;                 // row stride of out (elements)
  int n_out;               // valid output columns
  int b_rows;              // rows per expert in the B tensor(s)
  int K;                   // reduction length
  int Tk;                  // rows of A and out
  int E;
  int n_tiles;             // output column tiles per expert
  int* status;
  unsigned long long wait_ns;
};

// Waits that only drain work already issued (copies, MMAs) before the CTA
// exits never use a limit below this, whatever the caller's wait limit.
constexpr uint64_t kDrainFloorNs = 2000000000ull;

__device__ __forceinline__ uint64_t drain_limit(uint64_t wait_ns) {
  return wait_ns > kDrainFloorNs ? wait_ns : kDrainFloorNs;
}

__device__ __forceinline__ void raise_abort(SmemCtl* ctl, int* status) {
  *reinterpret_cast<volatile int*>(&ctl->abort_flag) = 1;
  record_status(status, MOE_ETIMEOUT);
}

__device__ __forceinline__ void decode_tile(const SmemCtl* ctl, int E, int tile, int& e, int& m, int& n) {
  e = 0;
  while (e + 1 < E && ctl->tile_prefix[e + 1] <= tile) ++e;
  const int local = tile - ctl->tile_prefix[e];
  const int mt = ctl->mtiles[e];
  n = local / mt;
  m = local - n * mt;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Small batches: the routing kernels ahead of this one leave HBM idle for a
// few microseconds while this CTA is already resident (programmatic
// dependent launch).  If every expert has rows - at decode nearly always -
// this CTA's first tile is tile blockIdx.x of the full table: expert
// t / n_tiles, column block t % n_tiles.  Its weight rows do not depend on
// the kernels still running, so the first MOE_PREFETCH_ROW_BYTES of each are
// requested into L2 now, before the wait.  When the guess is wrong the bytes
// are fetched for nothing; nothing reads them wrongly.  bf16 weights only:
// on the decode layer 2 KB of each 8 KB row took 1.3% off the layer (more
// was slower); for int8 weights any amount made the layer slower.
template <bool SWIGLU>
__device__ __forceinline__ void prefetch_first_tile(const GemmArgs& args, int lane) {
  const int t = blockIdx.x;
  if (args.n_tiles <= 0 || t >= args.E * args.n_tiles) return;
  const int e = t / args.n_tiles;
  const int n = t - e * args.n_tiles;
  const size_t row_bytes = static_cast<size_t>(args.K) * static_cast<size_t>(args.b_esz);
  const size_t want = row_bytes < static_cast<size_t>(MOE_PREFETCH_ROW_BYTES) ? row_bytes
                                                                               : static_cast<size_t>(MOE_PREFETCH_ROW_BYTES);
  const uint32_t bytes = static_cast<uint32_t>(want) & ~15u;
  if (bytes == 0) return;
  for (int i = lane; i < BN; i += 32) {  // the tile's 256 weight rows
    const int r = SWIGLU ? n * BN_HALF + (i % BN_HALF) : n * BN + i;
    const uint8_t* base = (SWIGLU && i >= BN_HALF) ? args.b1 : args.b0;
    if (r < args.b_rows)
      ptx::prefetch_l2_bulk(base + (static_cast<size_t>(e) * args.b_rows + r) * row_bytes, bytes);
  }
}

// The warp's 32 rows x 32 bf16 columns (lane = row, pk[i] = columns 2i, 2i+1)
// to dst[r * ld + ...] for r < rows.  Each lane writes its 64-byte row into
// the warp's staging block as four 16-byte units (unit j of row r at unit
// j ^ ((r >> 1) & 3), so that a quarter-warp meets distinct banks); then every
// load/store instruction moves eight whole 64-byte rows, four lanes per row,
// instead of touching 32 rows at once.
__device__ __forceinline__ void warp_store_rows_bf16(uint32_t stg, const uint32_t (&pk)[16], __nv_bfloat16* dst,
                                                     size_t ld, int rows, int lane) {
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    ptx::sts128(stg + lane * 64 + ((j ^ sw) << 4), make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]));
  __syncwarp();
  const int sub = lane >> 2, u = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 8 * i + sub;
    const uint4 val = ptx::lds128(stg + r * 64 + ((u ^ ((r >> 1) & 3)) << 4));
    if (r < rows) *reinterpret_cast<uint4*>(dst + static_cast<size_t>(r) * ld + 8 * u) = val;
  }
  __syncwarp();
}

// What the training forward keeps for the backward of h = silu(a) b, formed
// in fp32 from the GEMM's fp32 a and b and rounded once to bf16:
// p = dh/da / dh = b silu'(a) = b s (1 + a (1 - s)) and q = dh/db / dh =
// silu(a) = a s, with s = sigmoid(a).  The backward then needs only
// da = dh p and db = dh q.
// e = exp(-a), shared with the h computation.
__device__ __forceinline__ void keep_pair(float a, float b, float e, float& p, float& q) {
  const float s = __frcp_rn(1.0f + e);
  q = a * s;
  p = b * (s * (1.0f + a * (1.0f - s)));
}

template <bool SWIGLU, bool W8, bool SWAP>
__global__ void __launch_bounds__(Plan<W8, SWAP>::threads, 1)
    grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                           const __grid_constant__ CUtensorMap tmB1, const GemmArgs args) {
  using P = Plan<W8, SWAP>;
  constexpr int NST = P::stages;
  constexpr int SB = P::stage_bytes;
  constexpr int AB = P::a_bytes;
  constexpr int ROWS = P::rows;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* toks = smem + NST * SB;  // int8: token ring
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem + P::ring_bytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const volatile int* abort_flag = &ctl->abort_flag;

  // Set-up that reads nothing the previous kernel writes: barriers, tensor
  // maps, tensor memory.  It overlaps the previous kernel's tail.
  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      ptx::mbar_init(&ctl->full[s], 1);
      ptx::mbar_init(&ctl->empty[s], W8 ? CONV_WARPS : 1);
    }
    // Barriers the MMAs complete get one arrival per issuing thread.
    for (int s = 0; s < P::tok_stages; ++s) {
      ptx::mbar_init(&ctl->tok_full[s], 1);
      ptx::mbar_init(&ctl->tok_empty[s], P::issuers);
    }
    for (int s = 0; s < (W8 ? TMEM_A_STAGES : 0); ++s) {
      ptx::mbar_init(&ctl->c_full[s], CONV_WARPS);
      ptx::mbar_init(&ctl->c_empty[s], P::issuers);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&ctl->tfull[a], P::issuers);
      ptx::mbar_init(&ctl->tempty[a], EPI_THREADS);
    }
    ptx::mbar_init(&ctl->drain, P::issuers);
    ctl->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB0);
    if (SWIGLU) ptx::prefetch_tmap(&tmB1);
  }
  if (warp == 1) {
    ptx::tmem_alloc(&ctl->tmem_base, P::tmem_cols);
    ptx::tmem_relinquish();
  }
  if (SWAP && !W8 && MOE_PREFETCH_ROW_BYTES > 0 && warp == 2) prefetch_first_tile<SWIGLU>(args, lane);
  pdl_enter();
  if (threadIdx.x == 0) {
    // Expert segments -> tile table.  A segment that is not inside [0, Tk]
    // or runs backwards is treated as empty and reported.
    int run = 0;
    int prev = 0;
    ctl->tile_prefix[0] = 0;
    for (int e = 0; e <= args.E; ++e) {
      int o = args.offsets[e];
      if (o < prev || o > args.Tk) {
        record_status(args.status, MOE_EDEVICE);
        o = prev;
      }
      ctl->seg[e] = o;
      prev = o;
    }
    for (int e = 0; e < args.E; ++e) {
      const int n_e = ctl->seg[e + 1] - ctl->seg[e];
      const int mt = (n_e + ROWS - 1) / ROWS;
      ctl->mtiles[e] = mt;
      run += mt * args.n_tiles;
      ctl->tile_prefix[e + 1] = run;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  const int total_tiles = ctl->tile_prefix[args.E];
  const int kblocks = (args.K + P::kstep - 1) / P::kstep;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      // bf16: A + both B boxes.  int8: A + both raw B boxes.
      int stage = 0;
      uint32_t phase = 0;
      uint32_t filled = 0;                // stages filled at least once
      uint32_t last_parity[MAX_STAGES];   // parity of each stage's latest fill
      for (int s = 0; s < MAX_STAGES; ++s) last_parity[s] = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        int e, m, n;
        decode_tile(ctl, args.E, tile, e, m, n);
        const int arow = ctl->seg[e] + m * ROWS;
        int b0row, b1row;
        if (SWIGLU) {
          b0row = e * args.b_rows + n * BN_HALF;
          b1row = b0row;
        } else {
          b0row = e * args.b_rows + n * BN;
          b1row = b0row + BN_HALF;
        }
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(&ctl->empty[stage], phase ^ 1u, abort_flag, args.wait_ns)) {
            raise_abort(ctl, args.status);
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * SB;
          constexpr int half = W8 ? RAW_W_HALF_BYTES : B_HALF_BYTES;
          const int k0 = kb * P::kstep;
          ptx::mbar_arrive_expect_tx(&ctl->full[stage], SB);
          if (!P::tmem_a) {
#pragma unroll
            for (int t = 0; t < P::kstep / BK; ++t)
              ptx::tma_load_2d(sa + t * P::tok_box_bytes, &tmA, &ctl->full[stage], k0 + t * BK, arow);
          }
          ptx::tma_load_2d(sa + P::b_off, &tmB0, &ctl->full[stage], k0, b0row);
          ptx::tma_load_2d(sa + P::b_off + half, SWIGLU ? &tmB1 : &tmB0, &ctl->full[stage], k0, b1row);
          filled |= 1u << stage;
          last_parity[stage] = phase;
          if (++stage == NST) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // No copy may still be writing shared memory when the CTA exits.
      for (int s = 0; s < NST; ++s) {
        if (filled & (1u << s)) ptx::mbar_wait(&ctl->full[s], last_parity[s], nullptr, drain_limit(args.wait_ns));
      }
    }
  } else if (warp == 1 || (P::issuers > 1 && warp == P::mma2_warp)) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      // int8: thread `half` issues the MMAs of its 128-row half only.
      const int half = warp == 1 ? 0 : 1;
      int stage = 0, cstage = 0;
      uint32_t phase = 0, cphase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        if (!ptx::mbar_wait(&ctl->tempty[acc], acc_phase ^ 1u, abort_flag, args.wait_ns)) {
          raise_abort(ctl, args.status);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * P::acc_cols);
        for (int kb = 0; kb < kblocks; ++kb) {
          // int8 swapped: the token ring (the weights arrive via c_full);
          // otherwise the operand stage.
          if (!ptx::mbar_wait(P::tmem_a ? &ctl->tok_full[stage] : &ctl->full[stage], phase, abort_flag,
                              args.wait_ns) ||
              (W8 && !ptx::mbar_wait(&ctl->c_full[cstage], cphase, abort_flag, args.wait_ns))) {
            raise_abort(ctl, args.status);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = P::tmem_a ? ptx::smem_u32(toks + stage * AB) : ptx::smem_u32(smem + stage * SB);
          const uint32_t sb = sa + AB;
          const uint32_t ta = tmem_base + TMEM_A_COL0 + static_cast<uint32_t>(cstage * TMEM_A_STAGE_COLS);
          if (SWAP) {
            // Small-batch forms: the operands' bases once per stage, constant
            // offsets per K step (descriptor start addresses count 16 bytes).
            const uint64_t tdesc0 = ptx::sdesc_kmajor_sw128(sa);
            const uint32_t acc0 = kb > 0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < P::kstep / UMMA_K; ++kk) {
              const uint32_t f = kk == 0 ? acc0 : 1u;
              // token operand: 64-wide box kk / 4, K offset (kk % 4) * 16 within it
              const uint64_t tdesc = tdesc0 + static_cast<uint64_t>(((kk / (BK / UMMA_K)) * P::tok_box_bytes +
                                                                      (kk % (BK / UMMA_K)) * UMMA_K * 2) >> 4);
              if (P::tmem_a) {
                // widened weights of this thread's half (128 lanes of tensor memory) x the 32-token tile
                ptx::umma_bf16_tmem_a(d_tmem + half * TN, ta + half * TMEM_A_HALF_COLS + kk * (UMMA_K / 2), tdesc,
                                      IDESC_SWAP, f);
              } else {
                // weights (two 128-row halves) x the 32-token tile
                const uint64_t w0 = ptx::sdesc_kmajor_sw128(sb) + static_cast<uint64_t>((kk * UMMA_K * 2) >> 4);
                const uint64_t w1 = w0 + static_cast<uint64_t>(B_HALF_BYTES >> 4);
                ptx::umma_bf16(d_tmem, w0, tdesc, IDESC_SWAP, f);
                ptx::umma_bf16(d_tmem + TN, w1, tdesc, IDESC_SWAP, f);
              }
            }
          } else {
            // Large batches: the 128-row token tile x 256 weight rows.
#pragma unroll
            for (int kk = 0; kk < P::kstep / UMMA_K; ++kk) {
              const uint32_t acc_flag = (kb > 0 || kk > 0) ? 1u : 0u;
              const uint64_t tdesc = ptx::sdesc_kmajor_sw128(sa + kk * UMMA_K * 2);
              const uint64_t bdesc = ptx::sdesc_kmajor_sw128(sb + kk * UMMA_K * 2);
              ptx::umma_bf16(d_tmem, tdesc, bdesc, IDESC, acc_flag);
            }
          }
          // frees the stage (int8 swapped: the token stage) once these MMAs are done
          ptx::umma_commit(P::tmem_a ? &ctl->tok_empty[stage] : &ctl->empty[stage]);
          if (W8) {
            ptx::umma_commit(&ctl->c_empty[cstage]);
            if (++cstage == TMEM_A_STAGES) {
              cstage = 0;
              cphase ^= 1u;
            }
          }
          if (++stage == (P::tmem_a ? P::tok_stages : NST)) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::umma_commit(&ctl->tfull[acc]);  // accumulator ready for the epilogue
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // Every MMA issued above must finish before TMEM is freed.
      ptx::umma_commit(&ctl->drain);
      ptx::mbar_wait(&ctl->drain, 0, nullptr, drain_limit(args.wait_ns));
    }
  } else if (warp < 6) {
    // -------------------------------------------------- epilogue (warps 2-5)
    const int quad = warp & 3;  // TMEM lanes this warp may read: 32*quad .. +31
    const int row_in_tile = quad * 32 + lane;
    constexpr bool scaled = W8;  // per-weight-row scales in the epilogue
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      int e, m, n;
      decode_tile(ctl, args.E, tile, e, m, n);
      // tcgen05.ld below is warp-collective: leave together or not at all.
      const bool ready = ptx::mbar_wait(&ctl->tfull[acc], acc_phase, abort_flag, args.wait_ns);
      if (!__all_sync(0xFFFFFFFFu, ready)) {
        raise_abort(ctl, args.status);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t t_row =
          tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * P::acc_cols);
      if (SWAP) {
        // Lane = weight row within a 128-row half; columns = the tile's tokens.
        const int row0 = ctl->seg[e] + m * TN;
        const int rows_here = min(TN, ctl->seg[e + 1] - row0);
#pragma unroll 1
        for (int hf = 0; hf < (SWIGLU ? 1 : 2); ++hf) {
          uint32_t a[32], b[32];
          ptx::tmem_ld_32x32b_x32(t_row + hf * TN, a);
          if (SWIGLU) ptx::tmem_ld_32x32b_x32(t_row + TN, b);
          ptx::tmem_ld_wait();
          const int col = SWIGLU ? n * BN_HALF + row_in_tile : n * BN + hf * BN_HALF + row_in_tile;
          if (col < args.n_out) {
            const size_t srow = static_cast<size_t>(e) * args.b_rows + col;
            const float s0 = scaled ? __ldg(args.scale0 + srow) : 1.0f;
            const float s1 = (scaled && SWIGLU) ? __ldg(args.scale1 + srow) : 1.0f;
            __nv_bfloat16* dst = args.out + static_cast<size_t>(row0) * args.ldo + col;
#pragma unroll
            for (int j = 0; j < TN; ++j) {
              if (j < rows_here) {
                float v = s0 * __uint_as_float(a[j]);
                if (SWIGLU) {
                  const float u = s1 * __uint_as_float(b[j]);
                  const float ev = __expf(-v);
                  if (!W8 && args.keep != nullptr) {
                    const size_t o = (static_cast<size_t>(row0) + j) * args.ldo + col;
                    float pp, qq;
                    keep_pair(v, u, ev, pp, qq);
                    args.keep[o] = __float2bfloat16_rn(pp);
                    args.keep[static_cast<size_t>(args.Tk) * args.ldo + o] = __float2bfloat16_rn(qq);
                  }
                  v = v / (1.0f + ev) * u;
                }
                dst[static_cast<size_t>(j) * args.ldo] = __float2bfloat16_rn(v);
              }
            }
          }
        }
      } else if (SWIGLU) {
        const int col0 = n * BN_HALF;
        const int wrow0 = ctl->seg[e] + m * ROWS + quad * 32;  // the warp's first row
        const int wrows = max(0, min(32, ctl->seg[e + 1] - wrow0));
        const uint32_t stg = ptx::smem_u32(smem + P::ring_bytes + P::ctl_bytes) + quad * 32 * 64;
#pragma unroll 1
        for (int c = 0; c < BN_HALF; c += 32) {
          uint32_t g[32], u[32];
          ptx::tmem_ld_32x32b_x32(t_row + c, g);
          ptx::tmem_ld_32x32b_x32(t_row + BN_HALF + c, u);
          ptx::tmem_ld_wait();
          if (col0 + c < args.n_out) {
            const size_t srow = static_cast<size_t>(e) * args.b_rows + col0 + c;
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
              float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
              if (scaled) {
                const float2 sg = __ldg(reinterpret_cast<const float2*>(args.scale0 + srow) + i);
                const float2 su = __ldg(reinterpret_cast<const float2*>(args.scale1 + srow) + i);
                g0 *= sg.x;
                g1 *= sg.y;
                u0 *= su.x;
                u1 *= su.y;
              }
              const float e0 = __expf(-g0), e1 = __expf(-g1);
              const float h0 = g0 / (1.0f + e0) * u0;
              const float h1 = g1 / (1.0f + e1) * u1;
              pk[i] = pack_bf16x2(h0, h1);
              if (!W8 && args.keep != nullptr) {
                // The training forward also keeps p and q (keep_pair) for the backward.
                float p0, q0, p1, q1;
                keep_pair(g0, u0, e0, p0, q0);
                keep_pair(g1, u1, e1, p1, q1);
                // In place: later iterations j > i read only g[2j], u[2j] (+1), past i.
                g[i] = pack_bf16x2(p0, p1);
                u[i] = pack_bf16x2(q0, q1);
              }
            }
            const size_t o = static_cast<size_t>(wrow0) * args.ldo + col0 + c;
            warp_store_rows_bf16(stg, pk, args.out + o, args.ldo, wrows, lane);
            if (!W8 && args.keep != nullptr) {
              uint32_t pp[16], qq[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                pp[i] = g[i];
                qq[i] = u[i];
              }
              warp_store_rows_bf16(stg, pp, args.keep + o, args.ldo, wrows, lane);
              warp_store_rows_bf16(stg, qq, args.keep + static_cast<size_t>(args.Tk) * args.ldo + o, args.ldo, wrows,
                                   lane);
            }
          }
        }
      } else {
        const int col0 = n * BN;
        const int wrow0 = ctl->seg[e] + m * ROWS + quad * 32;  // the warp's first row
        const int wrows = max(0, min(32, ctl->seg[e + 1] - wrow0));
        const uint32_t stg = ptx::smem_u32(smem + P::ring_bytes + P::ctl_bytes) + quad * 32 * 64;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(t_row + c, v);
          ptx::tmem_ld_wait();
          if (col0 + c < args.n_out) {
            const size_t srow = static_cast<size_t>(e) * args.b_rows + col0 + c;
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float y0 = __uint_as_float(v[2 * i]), y1 = __uint_as_float(v[2 * i + 1]);
              if (scaled) {
                const float2 sy = __ldg(reinterpret_cast<const float2*>(args.scale0 + srow) + i);
                y0 *= sy.x;
                y1 *= sy.y;
              }
              pk[i] = pack_bf16x2(y0, y1);
            }
            warp_store_rows_bf16(stg, pk, args.out + static_cast<size_t>(wrow0) * args.ldo + col0 + c, args.ldo, wrows,
                                 lane);
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&ctl->tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  } else if (P::tmem_a && warp == P::tok_warp) {
    if (lane == 0) {
      // ------------------------------------------------ token-tile producer (int8 swapped)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t filled = 0;
      uint32_t last_parity[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        int e, m, n;
        decode_tile(ctl, args.E, tile, e, m, n);
        const int arow = ctl->seg[e] + m * ROWS;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(&ctl->tok_empty[stage], phase ^ 1u, abort_flag, args.wait_ns)) {
            raise_abort(ctl, args.status);
            ok = false;
            break;
          }
          uint8_t* st = toks + stage * AB;
          ptx::mbar_arrive_expect_tx(&ctl->tok_full[stage], AB);
#pragma unroll
          for (int t = 0; t < P::kstep / BK; ++t)
            ptx::tma_load_2d(st + t * P::tok_box_bytes, &tmA, &ctl->tok_full[stage], kb * P::kstep + t * BK, arow);
          filled |= 1u << stage;
          last_parity[stage] = phase;
          if (++stage == P::tok_stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < P::tok_stages; ++s) {
        if (filled & (1u << s)) ptx::mbar_wait(&ctl->tok_full[s], last_parity[s], nullptr, drain_limit(args.wait_ns));
      }
    }
  } else if (W8) {
    // -------------------------------------------------- converters (int8, warps 6-13)
    // Warp q (= warp % 4) may access tensor-memory lanes 32q .. 32q+31: lane
    // r holds weight row r of each 128-row half, 128 K values as 64 columns.
    // The raw tile was stored with the 128-byte swizzle (16-byte unit u of
    // row r at unit u ^ (r % 8)), so the row reads of 8 lanes hit distinct
    // banks.  Group g takes the K steps c (counted over all of the CTA's
    // tiles) with c % CONV_GROUPS == g.  Per step: wait until the MMA is
    // done with the tensor-memory stage and the raw stage has landed, widen,
    // store, then mark the widened stage ready and release the raw stage.
    const uint32_t grp = static_cast<uint32_t>(warp - 6) / CONV_WARPS;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) + TMEM_A_COL0;
    uint32_t cnt = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
      for (int kb = 0; kb < kblocks; ++kb, ++cnt) {
        if (cnt % CONV_GROUPS != grp) continue;
        const int stage = static_cast<int>(cnt % NST);
        const uint32_t phase = (cnt / NST) & 1u;
        const int cstage = static_cast<int>(cnt % TMEM_A_STAGES);
        const uint32_t cphase = (cnt / TMEM_A_STAGES) & 1u;
        // Waits are warp-uniform: the warp goes on or leaves as one.
        const bool ready = ptx::mbar_wait(&ctl->c_empty[cstage], cphase ^ 1u, abort_flag, args.wait_ns) &&
                           ptx::mbar_wait(&ctl->full[stage], phase, abort_flag, args.wait_ns);
        if (!__all_sync(0xFFFFFFFFu, ready)) {
          raise_abort(ctl, args.status);
          ok = false;
          break;
        }
        const uint32_t rs = ptx::smem_u32(smem + stage * SB) + r * BK_W;
        const uint32_t tl = t_lane + static_cast<uint32_t>(cstage * TMEM_A_STAGE_COLS);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {  // 64 codes = 32 columns at a time
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
              v[u] = ptx::lds128(rs + hf * RAW_W_HALF_BYTES + (((4 * q + u) ^ (r & 7)) << 4));
            uint32_t w[32];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              i8x4_to_bf16x4(v[u].x, w[8 * u + 0], w[8 * u + 1]);
              i8x4_to_bf16x4(v[u].y, w[8 * u + 2], w[8 * u + 3]);
              i8x4_to_bf16x4(v[u].z, w[8 * u + 4], w[8 * u + 5]);
              i8x4_to_bf16x4(v[u].w, w[8 * u + 6], w[8 * u + 7]);
            }
            ptx::tmem_st_32x32b_x32(tl + hf * TMEM_A_HALF_COLS + q * 32, w);
          }
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(&ctl->c_full[cstage]);
          ptx::mbar_arrive(&ctl->empty[stage]);
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    ptx::tmem_dealloc(tmem_base, P::tmem_cols);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
    }
  });
  return fn;
}

// Row-major matrix [rows, inner] -> tensor map with 64 x box_rows boxes (128 x
// box_rows for wide int8) and zero fill outside the matrix.  bf16: 128-byte
// swizzle (the tcgen05 operand layout).  int8: 64-byte rows, unswizzled (read
// back 16 bytes per thread along rows), or 128-byte rows with the 128-byte
// swizzle (read back one row per thread).
int make_tmap(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, bool int8, int box_rows,
              bool wide_int8 = false) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return MOE_ECUDA;
  const uint64_t esz = int8 ? 1 : 2;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * esz};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(wide_int8 ? BK_W : BK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        (int8 && !wide_int8) ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ECUDA;
}

// Persistent grid size.  With many waves of tiles every SM is used.  With
// only a few waves (small batches, where the kernel streams weights and is
// bound by HBM), the last wave would leave most SMs idle while a few finish,
// so the grid is shrunk (to no fewer than 3/4 of the SMs) to the size that
// wastes the fewest tile slots in the last wave: 896 decode tiles run as
// 7 x 128 rather than 6 x 148 + 8.
int balanced_grid(long long tiles, int num_sms) {
  if (tiles <= num_sms) return static_cast<int>(tiles < 1 ? 1 : tiles);
  if (tiles >= 8LL * num_sms) return num_sms;
  int best = num_sms;
  long long best_waste = (tiles + num_sms - 1) / num_sms * num_sms - tiles;
  for (int g = num_sms - 1; g * 4 >= num_sms * 3; --g) {
    const long long waste = (tiles + g - 1) / g * g - tiles;
    if (waste < best_waste) {
      best = g;
      best_waste = waste;
    }
  }
  return best;
}

template <bool SWIGLU, bool W8, bool SWAP>
int smem_attr_once(int device) {
  static std::mutex mu;
  static bool done[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return MOE_ECUDA;
  if (!done[device]) {
    if (cudaFuncSetAttribute(grouped_gemm_tc_kernel<SWIGLU, W8, SWAP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(Plan<W8, SWAP>::smem_bytes)) != cudaSuccess) {
      return MOE_ECUDA;
    }
    done[device] = true;
  }
  return MOE_OK;
}

template <bool SWIGLU, bool W8, bool SWAP>
int launch_mode(const void* A, const void* B0, const void* B1, GemmArgs a, const Ctx& c, cudaStream_t s) {
  using P = Plan<W8, SWAP>;
  CUtensorMap ta, tb0, tb1;
  int rc = make_tmap(&ta, A, static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.Tk), false, P::rows);
  if (rc != MOE_OK) return rc;
  const uint64_t brows = static_cast<uint64_t>(a.E) * a.b_rows;
  rc = make_tmap(&tb0, B0, static_cast<uint64_t>(a.K), brows, W8, BN_HALF, P::tmem_a);
  if (rc != MOE_OK) return rc;
  if (SWIGLU) {
    rc = make_tmap(&tb1, B1, static_cast<uint64_t>(a.K), brows, W8, BN_HALF, P::tmem_a);
    if (rc != MOE_OK) return rc;
  } else {
    tb1 = tb0;
  }
  rc = smem_attr_once<SWIGLU, W8, SWAP>(c.device);
  if (rc != MOE_OK) return rc;
  // Upper bound on tiles: whole row blocks plus at most one partial block
  // per expert that has rows (at most min(E, Tk) of them); with a known
  // bound on any expert's rows (the layer passes T: a token picks an expert
  // at most once), also E times that bound's blocks.  The grid is sized
  // from it, so a tight bound avoids a nearly empty last wave.
  long long blocks = static_cast<long long>(a.Tk) / P::rows + (a.E < a.Tk ? a.E : a.Tk);
  if (c.max_rows_per_expert > 0) {
    const long long per = (static_cast<long long>(c.max_rows_per_expert < a.Tk ? c.max_rows_per_expert : a.Tk) +
                           P::rows - 1) / P::rows;
    if (per * a.E < blocks) blocks = per * a.E;
  }
  const long long max_tiles = blocks * static_cast<long long>(a.n_tiles);
  const int grid = balanced_grid(max_tiles, c.num_sms);
  launch_pdl(grouped_gemm_tc_kernel<SWIGLU, W8, SWAP>, grid, P::threads, P::smem_bytes, s, ta, tb0, tb1, a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ECUDA;
}

template <bool SWIGLU, bool W8>
int launch_gemm(const void* A, const void* B0, const void* B1, const float* S0, const float* S1,
                const int32_t* offsets, void* out, int Tk, int K, int n_out, int b_rows, int E, const Ctx& c,
                cudaStream_t s, void* keep = nullptr) {
  if (Tk <= 0) return MOE_OK;
  GemmArgs a;
  a.offsets = offsets;
  a.b0 = static_cast<const uint8_t*>(B0);
  a.b1 = static_cast<const uint8_t*>(B1);
  a.b_esz = W8 ? 1 : 2;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.keep = static_cast<__nv_bfloat16*>(keep);
  a.scale0 = S0;
  a.scale1 = S1;
  a.ldo = n_out;
  a.n_out = n_out;
  a.b_rows = b_rows;
  a.K = K;
  a.Tk = Tk;
  a.E = E;
  a.n_tiles = SWIGLU ? (n_out + BN_HALF - 1) / BN_HALF : (n_out + BN - 1) / BN;
  a.status = c.status;
  a.wait_ns = c.wait_ns;
  // Few rows (decode): weights as the MMA's M operand, 32 tokens as N.  The
  // int8 weights come here only with few rows (more go to the wide kernel).
  if constexpr (W8) {
    return launch_mode<SWIGLU, true, true>(A, B0, B1, a, c, s);
  } else {
    if (Tk <= SWAP_MAX_ROWS) return launch_mode<SWIGLU, false, true>(A, B0, B1, a, c, s);
    return launch_mode<SWIGLU, false, false>(A, B0, B1, a, c, s);
  }
}

}  // namespace

int launch_tc_gate_up(const void* x_perm, const int32_t* offsets, const void* W1, const void* W3, void* h, int Tk,
                      int d, int dff, int E, const Ctx& c, cudaStream_t s, void* keep) {
  return launch_gemm<true, false>(x_perm, W1, W3, nullptr, nullptr, offsets, h, Tk, d, dff, dff, E, c, s, keep);
}

int launch_tc_down(const void* h, const int32_t* offsets, const void* W2, void* y, int Tk, int d, int dff, int E,
                   const Ctx& c, cudaStream_t s) {
  return launch_gemm<false, false>(h, W2, nullptr, nullptr, nullptr, offsets, y, Tk, dff, d, d, E, c, s);
}

int launch_w8_gate_up(const void* x_perm, const int32_t* offsets, const int8_t* W1q, const float* W1s,
                      const int8_t* W3q, const float* W3s, void* h, int Tk, int d, int dff, int E, const Ctx& c,
                      cudaStream_t s) {
  if (Tk > SWAP_MAX_ROWS) return launch_w8_wide_gate_up(x_perm, offsets, W1q, W1s, W3q, W3s, h, Tk, d, dff, E, c, s);
  return launch_gemm<true, true>(x_perm, W1q, W3q, W1s, W3s, offsets, h, Tk, d, dff, dff, E, c, s);
}

int launch_w8_down(const void* h, const int32_t* offsets, const int8_t* W2q, const float* W2s, void* y, int Tk, int d,
                   int dff, int E, const Ctx& c, cudaStream_t s) {
  if (Tk > SWAP_MAX_ROWS) return launch_w8_wide_down(h, offsets, W2q, W2s, y, Tk, d, dff, E, c, s);
  return launch_gemm<false, true>(h, W2q, nullptr, W2s, nullptr, offsets, y, Tk, dff, d, d, E, c, s);
}

}  // namespace moe
