// Steps a4-a5 with int8 weight-only experts beyond the small-batch case
// ("The Evolving Transformer - 05 Mixtral", section 04 SwiGLU; KerasFormers
// Mixtral docs, "Lower memory": the weights alone quantised to int8, one fp32
// scale per output row, activations in bf16).
//
// The weights stream as int8 and are widened on the SM.  Widened in shared
// memory, a 128-row token tile x 256 weight rows costs more shared-memory
// traffic than the tensor cores leave room for; widened once per call into a
// bf16 copy in HBM, they cost 4.2 GB of extra traffic.  Here they are widened
// straight into tensor memory, where the MMA takes them as its A operand, and
// every widened weight row meets 224 tokens:
//   tile     128 weight rows (the MMA's M, tensor-memory lanes) x 224 tokens
//            of one expert's segment (the MMA's N, K-major from shared
//            memory).  Gate/up: rows 0-63 are W1 rows f0..f0+63 and rows
//            64-127 the W3 rows of the same hidden units, so one accumulator
//            holds both halves of the SwiGLU; down: 128 rows of W2.
//   warp 0   TMA producer: per 64-deep K step the 224 x 64 bf16 token box
//            (128-byte swizzle) and the 128 x 64 int8 weight rows (64-byte
//            swizzle) into a 5-stage ring.
//   warps 6-13 converters, two groups of four taking alternate K steps (a
//            group's step is a chain of shared-memory loads, widening, a
//            tensor-memory store and its wait; two groups overlap those
//            chains): lane r of warp q (q = warp % 4, the tensor-memory lane
//            quarter it may write) widens weight row r = 32q + lane of the
//            stage - 64 codes, exactly - and writes it to tensor memory
//            (tcgen05.st, two bf16 per 32-bit column) in a 2-deep ring of A
//            stages; a raw stage is free once the MMA has read the tokens and
//            the group's converters the weights.
//   warp 1   tensor memory (512 columns: two 224-column accumulators and the
//            A ring) and tcgen05.mma kind::f16, M=128, N=224, K=16, A from
//            tensor memory; the two accumulators alternate between tiles so
//            the epilogue of one overlaps the MMAs of the next.
//   warps 2-5 epilogue: the accumulator times the weight row's scale.  Down:
//            each lane owns one output column for the tile's 224 tokens.
//            Gate/up: per 32-token chunk, the warps holding the W1 rows and
//            those holding the W3 rows of the same hidden units swap half of
//            their scaled values through shared memory, so that all four
//            warps form h = silu(gate) * up for 16 tokens each and store it.
// The widening and the MMAs share the tensor memory; a tile of 224 tokens
// makes every expert of the T=4096 Mixtral batch (1000-1036 routed rows)
// five tiles, so each weight is widened five times per call.
// Tiles are numbered expert by expert, weight block slowest and token tile
// fastest, so the CTAs running at one time share each weight block through
// L2.  An expert with no rows has no tiles.  Every wait is bounded; a wait
// that runs out raises a CTA-wide abort flag and records MOE_ETIMEOUT, the
// roles leave their loops, drain what they issued and free tensor memory.
#include <cuda.h>
#include <mutex>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "widen.cuh"

namespace moe {
namespace {

constexpr int WM = 128;                        // weight rows per tile (MMA M)
constexpr int WN = 224;                        // tokens per tile (MMA N)
constexpr int WK = 64;                         // K per stage
constexpr int UK = 16;                         // K per MMA
constexpr int STAGES = 5;
constexpr int TOK_BYTES = WN * WK * 2;         // 24 KB token box
constexpr int RAW_BYTES = WM * WK;             // 8 KB of int8 weight rows (64-byte rows)
constexpr int STAGE_BYTES = TOK_BYTES + RAW_BYTES;
constexpr int A_STAGES = 2;
constexpr int A_COLS = WK / 2;                 // 32-bit columns of one widened K step
constexpr int ACC_COLS = WN;
constexpr int A_COL0 = 2 * ACC_COLS;
constexpr int TMEM_COLS = 512;
constexpr int CONV_WARPS = 4;                  // one per tensor-memory lane quarter
constexpr int CONV_GROUPS = 2;                 // groups of CONV_WARPS, taking alternate K steps
constexpr int THREADS = 192 + 32 * CONV_WARPS * CONV_GROUPS;
constexpr int EPI_THREADS = 128;
constexpr int HALF = WM / 2;                   // gate/up: hidden units per tile
constexpr int XCH_WORDS = 32 * HALF;           // one 32-token chunk: 16 tokens of gate + 16 of up values
constexpr int MAX_E = 64;
constexpr uint32_t IDESC = ptx::idesc_bf16_f32(WM, WN);
static_assert(A_COL0 + A_STAGES * A_COLS <= TMEM_COLS, "tensor memory: accumulators + A ring");
static_assert(WN % 16 == 0 && WN <= 256, "MMA N");
static_assert(WN % 32 == 0, "epilogue chunks of 32 tokens");

struct Ctl {
  uint64_t full[STAGES];      // the stage's token box and weight rows landed
  uint64_t empty[STAGES];     // the MMA (tokens) and every converter (weights) are done with it
  uint64_t a_full[A_STAGES];  // widened weights written to tensor memory
  uint64_t a_empty[A_STAGES]; // the MMA is done with them
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int tile_prefix[MAX_E + 1];
  int mtiles[MAX_E];
  int seg[MAX_E + 1];
};

constexpr size_t SMEM_BYTES = 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + 2 * XCH_WORDS * sizeof(float) +
                              sizeof(Ctl);
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per block");

struct WideArgs {
  const int32_t* offsets;  // [E+1], device
  __nv_bfloat16* out;      // [Tk, n_out]
  const float* scale0;     // row scales of W1 (gate/up) or W2 (down), [E * b_rows]
  const float* scale1;     // row scales of W3 (gate/up)
  int n_out;               // output columns: dff (gate/up) or d (down)
  int b_rows;              // rows per expert of each weight tensor
  int K;                   // reduction length: d (gate/up) or dff (down)
  int Tk;
  int E;
  int n_tiles;             // weight blocks per expert
  int* status;
  unsigned long long wait_ns;
};

constexpr uint64_t kDrainFloorNs = 2000000000ull;
__device__ __forceinline__ uint64_t drain_limit(uint64_t w) { return w > kDrainFloorNs ? w : kDrainFloorNs; }

__device__ __forceinline__ void raise_abort(Ctl* ctl, int* status) {
  *reinterpret_cast<volatile int*>(&ctl->abort_flag) = 1;
  record_status(status, MOE_ETIMEOUT);
}

__device__ __forceinline__ void decode_tile(const Ctl* ctl, int E, int tile, int& e, int& m, int& n) {
  e = 0;
  while (e + 1 < E && ctl->tile_prefix[e + 1] <= tile) ++e;
  const int local = tile - ctl->tile_prefix[e];
  const int mt = ctl->mtiles[e];
  n = local / mt;
  m = local - n * mt;
}

// Named barrier 1 over the four epilogue warps; returns the AND of `pred`
// over them.
__device__ __forceinline__ bool epi_all(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred))
      : "memory");
  return r != 0;
}

// Named barrier 2 over the four epilogue warps.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

template <bool SWIGLU>
__global__ void __launch_bounds__(THREADS, 1)
    w8_wide_gemm_kernel(const __grid_constant__ CUtensorMap tmT, const __grid_constant__ CUtensorMap tmW0,
                        const __grid_constant__ CUtensorMap tmW1, const WideArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* xch = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + STAGES * STAGE_BYTES + 2 * XCH_WORDS * sizeof(float));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const volatile int* abort_flag = &ctl->abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&ctl->full[s], 1);
      ptx::mbar_init(&ctl->empty[s], 1 + CONV_WARPS);
    }
    for (int s = 0; s < A_STAGES; ++s) {
      ptx::mbar_init(&ctl->a_full[s], CONV_WARPS);
      ptx::mbar_init(&ctl->a_empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&ctl->tfull[a], 1);
      ptx::mbar_init(&ctl->tempty[a], EPI_THREADS);
    }
    ptx::mbar_init(&ctl->drain, 1);
    ctl->abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmT);
    ptx::prefetch_tmap(&tmW0);
    if (SWIGLU) ptx::prefetch_tmap(&tmW1);
  }
  if (warp == 1) {
    ptx::tmem_alloc(&ctl->tmem_base, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  pdl_enter();
  if (threadIdx.x == 0) {
    // Expert segments -> tile table; a segment outside [0, Tk] or running
    // backwards is treated as empty and reported.
    int run = 0, prev = 0;
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
      const int mt = (ctl->seg[e + 1] - ctl->seg[e] + WN - 1) / WN;
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
  const int kblocks = args.K / WK;  // K is a multiple of 64 (host-checked)

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0, filled = 0;
      uint32_t last_parity[STAGES];
      for (int s = 0; s < STAGES; ++s) last_parity[s] = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        int e, m, n;
        decode_tile(ctl, args.E, tile, e, m, n);
        const int arow = ctl->seg[e] + m * WN;
        const int wrow = e * args.b_rows + n * (SWIGLU ? HALF : WM);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(&ctl->empty[stage], phase ^ 1u, abort_flag, args.wait_ns)) {
            raise_abort(ctl, args.status);
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * STAGE_BYTES;
          const int k0 = kb * WK;
          ptx::mbar_arrive_expect_tx(&ctl->full[stage], STAGE_BYTES);
          ptx::tma_load_2d(sa, &tmT, &ctl->full[stage], k0, arow);
          ptx::tma_load_2d(sa + TOK_BYTES, &tmW0, &ctl->full[stage], k0, wrow);
          if (SWIGLU) ptx::tma_load_2d(sa + TOK_BYTES + HALF * WK, &tmW1, &ctl->full[stage], k0, wrow);
          filled |= 1u << stage;
          last_parity[stage] = phase;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < STAGES; ++s)
        if (filled & (1u << s)) ptx::mbar_wait(&ctl->full[s], last_parity[s], nullptr, drain_limit(args.wait_ns));
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int stage = 0, cs = 0, acc = 0;
      uint32_t phase = 0, cphase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        if (!ptx::mbar_wait(&ctl->tempty[acc], acc_phase ^ 1u, abort_flag, args.wait_ns)) {
          raise_abort(ctl, args.status);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * ACC_COLS);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(&ctl->full[stage], phase, abort_flag, args.wait_ns) ||
              !ptx::mbar_wait(&ctl->a_full[cs], cphase, abort_flag, args.wait_ns)) {
            raise_abort(ctl, args.status);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t tok = ptx::smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t ta = tmem_base + static_cast<uint32_t>(A_COL0 + cs * A_COLS);
#pragma unroll
          for (int kk = 0; kk < WK / UK; ++kk) {
            const uint64_t bdesc = ptx::sdesc_kmajor_sw128(tok + kk * UK * 2);
            ptx::umma_bf16_tmem_a(d_tmem, ta + kk * (UK / 2), bdesc, IDESC, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::umma_commit(&ctl->empty[stage]);
          ptx::umma_commit(&ctl->a_empty[cs]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if (++cs == A_STAGES) {
            cs = 0;
            cphase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::umma_commit(&ctl->tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      ptx::umma_commit(&ctl->drain);
      ptx::mbar_wait(&ctl->drain, 0, nullptr, drain_limit(args.wait_ns));
    }
  } else if (warp < 6) {
    // -------------------------------------------------- epilogue (warps 2-5)
    const int quad = warp & 3;  // tensor-memory lanes 32*quad .. +31
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      int e, m, n;
      decode_tile(ctl, args.E, tile, e, m, n);
      const int row0 = ctl->seg[e] + m * WN;
      const int rows_here = min(WN, ctl->seg[e + 1] - row0);
      bool ready = ptx::mbar_wait(&ctl->tfull[acc], acc_phase, abort_flag, args.wait_ns);
      ready = __all_sync(0xFFFFFFFFu, ready);
      // All four warps go on, or all leave: the gate/up epilogue meets at a
      // named barrier once per chunk.
      if (!epi_all(ready)) {
        raise_abort(ctl, args.status);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t t_lane =
          tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * ACC_COLS);
      if (SWIGLU) {
        // Lanes 0-63: gate rows (W1) of hidden units f0 .. f0+63; lanes
        // 64-127: up rows (W3) of the same units.  Per chunk of 32 tokens the
        // gate warps take tokens 0-15 and the up warps tokens 16-31; each
        // side hands the other the scaled values of the other's tokens.
        const bool up = quad >= 2;
        const int fl = (quad & 1) * 32 + lane;
        const int f = n * HALF + fl;
        const size_t srow = static_cast<size_t>(e) * args.b_rows + f;
        const float s = __ldg((up ? args.scale1 : args.scale0) + srow);
        const int i0 = up ? 16 : 0;  // this warp's tokens within a chunk
        __nv_bfloat16* dst = args.out + static_cast<size_t>(row0) * args.n_out + f;
#pragma unroll 1
        for (int c = 0; c < WN / 32; ++c) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(t_lane + c * 32, v);
          ptx::tmem_ld_wait();
          float* xb = xch + (c & 1) * XCH_WORDS;   // [0, 16*HALF): gate values; then up values
          float* mine = xb + (up ? 16 * HALF : 0);  // where this side leaves the other's tokens
          const float* theirs = xb + (up ? 0 : 16 * HALF);
          // (Register indices stay compile-time: the side is picked by branch.)
          if (up) {
#pragma unroll
            for (int i = 0; i < 16; ++i) mine[i * HALF + fl] = s * __uint_as_float(v[i]);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) mine[i * HALF + fl] = s * __uint_as_float(v[16 + i]);
          }
          epi_sync();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int j = c * 32 + i0 + i;
            if (j < rows_here) {
              const float own = s * __uint_as_float(up ? v[16 + i] : v[i]);
              const float other = theirs[i * HALF + fl];
              const float g = up ? other : own;
              const float u = up ? own : other;
              const float hv = g * __frcp_rn(1.0f + __expf(-g)) * u;
              dst[static_cast<size_t>(j) * args.n_out] = __float2bfloat16_rn(hv);
            }
          }
        }
      } else {
        const int col = n * WM + quad * 32 + lane;
        const bool col_ok = col < args.n_out;
        const float s = col_ok ? __ldg(args.scale0 + static_cast<size_t>(e) * args.b_rows + col) : 0.0f;
        __nv_bfloat16* dst = args.out + static_cast<size_t>(row0) * args.n_out + col;
#pragma unroll 1
        for (int c = 0; c < WN / 32; ++c) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(t_lane + c * 32, v);
          ptx::tmem_ld_wait();
          if (col_ok) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int j = c * 32 + i;
              if (j < rows_here) dst[static_cast<size_t>(j) * args.n_out] = __float2bfloat16_rn(s * __uint_as_float(v[i]));
            }
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
  } else {
    // -------------------------------------------------- converters (warps 6-13)
    // Row r of the stage's weights -> tensor-memory lane r.  The rows are
    // 64 bytes under the 64-byte swizzle: 16-byte unit u of row r sits at
    // unit u ^ ((r >> 1) & 3), so the reads of eight consecutive lanes hit
    // distinct banks.  Group g takes the K steps q (counted over all of the
    // CTA's tiles) with q % CONV_GROUPS == g.
    const int quad = warp & 3;
    const uint32_t grp = static_cast<uint32_t>(warp - 6) / CONV_WARPS;
    const int r = quad * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(A_COL0);
    const int sw = (r >> 1) & 3;
    uint32_t q = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
      for (int kb = 0; kb < kblocks; ++kb, ++q) {
        if (q % CONV_GROUPS != grp) continue;
        const int stage = static_cast<int>(q % STAGES);
        const uint32_t phase = (q / STAGES) & 1u;
        const int cs = static_cast<int>(q % A_STAGES);
        const uint32_t cphase = (q / A_STAGES) & 1u;
        const bool ready = ptx::mbar_wait(&ctl->a_empty[cs], cphase ^ 1u, abort_flag, args.wait_ns) &&
                           ptx::mbar_wait(&ctl->full[stage], phase, abort_flag, args.wait_ns);
        if (!__all_sync(0xFFFFFFFFu, ready)) {
          raise_abort(ctl, args.status);
          ok = false;
          break;
        }
        const uint32_t rs = ptx::smem_u32(smem + stage * STAGE_BYTES + TOK_BYTES) + static_cast<uint32_t>(r * WK);
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = ptx::lds128(rs + static_cast<uint32_t>((u ^ sw) << 4));
        uint32_t w[32];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          i8x4_to_bf16x4(v[u].x, w[8 * u + 0], w[8 * u + 1]);
          i8x4_to_bf16x4(v[u].y, w[8 * u + 2], w[8 * u + 3]);
          i8x4_to_bf16x4(v[u].z, w[8 * u + 4], w[8 * u + 5]);
          i8x4_to_bf16x4(v[u].w, w[8 * u + 6], w[8 * u + 7]);
        }
        ptx::tmem_st_32x32b_x32(t_lane + static_cast<uint32_t>(cs * A_COLS), w);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(&ctl->a_full[cs]);
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
    ptx::tmem_dealloc(tmem_base, TMEM_COLS);
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

// Row-major [rows, inner] -> boxes of 64 inner elements x box_rows rows, zero
// fill outside the matrix: bf16 tokens with the 128-byte swizzle (tcgen05's
// K-major operand layout), int8 weight rows (64 bytes) with the 64-byte one.
int make_tmap(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, bool int8, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return MOE_ECUDA;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * (int8 ? 1 : 2)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(WK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        int8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ECUDA;
}

template <bool SWIGLU>
int smem_attr_once(int device) {
  static std::mutex mu;
  static bool done[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return MOE_ECUDA;
  if (!done[device]) {
    if (cudaFuncSetAttribute(w8_wide_gemm_kernel<SWIGLU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES)) != cudaSuccess)
      return MOE_ECUDA;
    done[device] = true;
  }
  return MOE_OK;
}

template <bool SWIGLU>
int launch_wide(const void* A, const int8_t* B0, const int8_t* B1, WideArgs a, const Ctx& c, cudaStream_t s) {
  if (a.Tk <= 0) return MOE_OK;
  CUtensorMap tt, t0, t1;
  const uint64_t brows = static_cast<uint64_t>(a.E) * a.b_rows;
  const int box = SWIGLU ? HALF : WM;
  int rc = make_tmap(&tt, A, static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.Tk), false, WN);
  if (rc == MOE_OK) rc = make_tmap(&t0, B0, static_cast<uint64_t>(a.K), brows, true, box);
  if (rc == MOE_OK) rc = SWIGLU ? make_tmap(&t1, B1, static_cast<uint64_t>(a.K), brows, true, box) : MOE_OK;
  if (rc != MOE_OK) return rc;
  if (!SWIGLU) t1 = t0;
  rc = smem_attr_once<SWIGLU>(c.device);
  if (rc != MOE_OK) return rc;
  a.status = c.status;
  a.wait_ns = c.wait_ns;
  // Upper bound on tiles (whole token tiles plus one partial tile per expert
  // that has rows, or E times the tiles of the known bound on any expert's
  // rows), for the persistent grid.
  long long blocks = static_cast<long long>(a.Tk) / WN + (a.E < a.Tk ? a.E : a.Tk);
  if (c.max_rows_per_expert > 0) {
    const long long per = (static_cast<long long>(c.max_rows_per_expert < a.Tk ? c.max_rows_per_expert : a.Tk) +
                           WN - 1) / WN;
    if (per * a.E < blocks) blocks = per * a.E;
  }
  const long long tiles = blocks * a.n_tiles;
  const int grid = static_cast<int>(tiles < c.num_sms ? (tiles < 1 ? 1 : tiles) : c.num_sms);
  launch_pdl(w8_wide_gemm_kernel<SWIGLU>, grid, THREADS, SMEM_BYTES, s, tt, t0, t1, a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ECUDA;
}

}  // namespace

int launch_w8_wide_gate_up(const void* x_perm, const int32_t* offsets, const int8_t* W1q, const float* W1s,
                           const int8_t* W3q, const float* W3s, void* h, int Tk, int d, int dff, int E, const Ctx& c,
                           cudaStream_t s) {
  WideArgs a = {};
  a.offsets = offsets;
  a.out = static_cast<__nv_bfloat16*>(h);
  a.scale0 = W1s;
  a.scale1 = W3s;
  a.n_out = dff;
  a.b_rows = dff;
  a.K = d;
  a.Tk = Tk;
  a.E = E;
  a.n_tiles = dff / HALF;
  return launch_wide<true>(x_perm, W1q, W3q, a, c, s);
}

int launch_w8_wide_down(const void* h, const int32_t* offsets, const int8_t* W2q, const float* W2s, void* y, int Tk,
                        int d, int dff, int E, const Ctx& c, cudaStream_t s) {
  WideArgs a = {};
  a.offsets = offsets;
  a.out = static_cast<__nv_bfloat16*>(y);
  a.scale0 = W2s;
  a.scale1 = nullptr;
  a.n_out = d;
  a.b_rows = d;
  a.K = dff;
  a.Tk = Tk;
  a.E = E;
  a.n_tiles = (d + WM - 1) / WM;
  return launch_wide<false>(h, W2q, nullptr, a, c, s);
}

}  // namespace moe
