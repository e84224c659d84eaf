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
//               bf16 rounding, stores of the rows that belong to the expert.
// Output tiles are 128 rows of one expert's segment x (gate/up) 128 columns
// of h, whose accumulator holds the W1 half in columns 0-127 and the W3 half
// in 128-255, or (down) 256 columns of y.  Tiles are numbered expert by
// expert, row block fastest, so CTAs running at the same time share the
// weight tile through L2.  Experts with no rows have no tiles, so their
// weights are never read.  The expert boundaries come from the device-side
// offsets[E+1]; the host never reads the per-expert counts.
//
// Every wait is bounded (globaltimer + iteration cap).  A wait that runs out
// raises a CTA-wide abort flag and records MOE_ETIMEOUT; each role then
// leaves its loop, the producer waits (bounded) for its copies in flight, the
// MMA warp waits (bounded) for its MMAs, and TMEM is freed before returning.
//
// The set-up (barriers, tensor-map prefetch, TMEM allocation) runs before the
// kernel waits on its predecessor (programmatic dependent launch), so it
// overlaps the previous kernel's tail.
#include <cuda.h>
#include <mutex>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;                  // rows (tokens) per tile
constexpr int BK = 64;                   // K per stage: one 128-byte swizzle row
constexpr int BN_HALF = 128;             // rows of one B box
constexpr int BN = 2 * BN_HALF;          // MMA N
constexpr int UMMA_K = 16;               // K of one tcgen05.mma (bf16)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;     // 16 KB
constexpr int B_HALF_BYTES = BN_HALF * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + 2 * B_HALF_BYTES;  // 48 KB
constexpr int TMEM_COLS = 2 * BN;        // two fp32 accumulators
constexpr int NUM_THREADS = 192;
constexpr int EPI_THREADS = 128;
constexpr int MAX_E = 64;
constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, BN);

struct SmemCtl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int tile_prefix[MAX_E + 1];
  int mtiles[MAX_E];
  int seg[MAX_E + 1];
};

constexpr size_t SMEM_BYTES = 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + sizeof(SmemCtl);

struct GemmArgs {
  const int32_t* offsets;  // [E+1], device
  __nv_bfloat16* out;      // [Tk, ldo]
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

__device__ __forceinline__ void decode_tile(const SmemCtl* ctl, int E, int n_tiles, int tile, int& e, int& m, int& n) {
  e = 0;
  while (e + 1 < E && ctl->tile_prefix[e + 1] <= tile) ++e;
  const int local = tile - ctl->tile_prefix[e];
  const int mt = ctl->mtiles[e];
  n = local / mt;
  m = local - n * mt;
  (void)n_tiles;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <bool SWIGLU>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                           const __grid_constant__ CUtensorMap tmB1, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem + STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const volatile int* abort_flag = &ctl->abort_flag;

  // Set-up that reads nothing the previous kernel writes: barriers, tensor
  // maps, tensor memory.  It overlaps the previous kernel's tail.
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&ctl->full[s], 1);
      ptx::mbar_init(&ctl->empty[s], 1);
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
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB0);
    if (SWIGLU) ptx::prefetch_tmap(&tmB1);
  }
  if (warp == 1) {
    ptx::tmem_alloc(&ctl->tmem_base, TMEM_COLS);
    ptx::tmem_relinquish();
  }
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
      const int mt = (n_e + BM - 1) / BM;
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
  const int kblocks = (args.K + BK - 1) / BK;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t filled = 0;            // stages filled at least once
      uint32_t last_parity[STAGES];   // parity of each stage's latest fill
      for (int s = 0; s < STAGES; ++s) last_parity[s] = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        int e, m, n;
        decode_tile(ctl, args.E, args.n_tiles, tile, e, m, n);
        const int arow = ctl->seg[e] + m * BM;
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
          uint8_t* sa = smem + stage * STAGE_BYTES;
          ptx::mbar_arrive_expect_tx(&ctl->full[stage], STAGE_BYTES);
          ptx::tma_load_2d(sa, &tmA, &ctl->full[stage], kb * BK, arow);
          ptx::tma_load_2d(sa + A_BYTES, &tmB0, &ctl->full[stage], kb * BK, b0row);
          ptx::tma_load_2d(sa + A_BYTES + B_HALF_BYTES, SWIGLU ? &tmB1 : &tmB0, &ctl->full[stage], kb * BK, b1row);
          filled |= 1u << stage;
          last_parity[stage] = phase;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // No copy may still be writing shared memory when the CTA exits.
      for (int s = 0; s < STAGES; ++s) {
        if (filled & (1u << s)) ptx::mbar_wait(&ctl->full[s], last_parity[s], nullptr, drain_limit(args.wait_ns));
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        if (!ptx::mbar_wait(&ctl->tempty[acc], acc_phase ^ 1u, abort_flag, args.wait_ns)) {
          raise_abort(ctl, args.status);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait(&ctl->full[stage], phase, abort_flag, args.wait_ns)) {
            raise_abort(ctl, args.status);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            const uint64_t adesc = ptx::sdesc_kmajor_sw128(sa + kk * UMMA_K * 2);
            const uint64_t bdesc = ptx::sdesc_kmajor_sw128(sb + kk * UMMA_K * 2);
            ptx::umma_bf16(d_tmem, adesc, bdesc, IDESC, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::umma_commit(&ctl->empty[stage]);  // frees the stage once these MMAs are done
          if (++stage == STAGES) {
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
  } else {
    // -------------------------------------------------- epilogue (warps 2-5)
    const int quad = warp & 3;  // TMEM lanes this warp may read: 32*quad .. +31
    const int row_in_tile = quad * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      int e, m, n;
      decode_tile(ctl, args.E, args.n_tiles, tile, e, m, n);
      const int grow = ctl->seg[e] + m * BM + row_in_tile;
      const bool row_ok = grow < ctl->seg[e + 1];
      // tcgen05.ld below is warp-collective: leave together or not at all.
      const bool ready = ptx::mbar_wait(&ctl->tfull[acc], acc_phase, abort_flag, args.wait_ns);
      if (!__all_sync(0xFFFFFFFFu, ready)) {
        raise_abort(ctl, args.status);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN);
      if (SWIGLU) {
        const int col0 = n * BN_HALF;
#pragma unroll 1
        for (int c = 0; c < BN_HALF; c += 32) {
          uint32_t g[32], u[32];
          ptx::tmem_ld_32x32b_x32(t_row + c, g);
          ptx::tmem_ld_32x32b_x32(t_row + BN_HALF + c, u);
          ptx::tmem_ld_wait();
          if (row_ok && col0 + c < args.n_out) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
              const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
              const float h0 = g0 / (1.0f + __expf(-g0)) * u0;
              const float h1 = g1 / (1.0f + __expf(-g1)) * u1;
              pk[i] = pack_bf16x2(h0, h1);
            }
            uint4* dst = reinterpret_cast<uint4*>(args.out + static_cast<size_t>(grow) * args.ldo + col0 + c);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
      } else {
        const int col0 = n * BN;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(t_row + c, v);
          ptx::tmem_ld_wait();
          if (row_ok && col0 + c < args.n_out) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
            uint4* dst = reinterpret_cast<uint4*>(args.out + static_cast<size_t>(grow) * args.ldo + col0 + c);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
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

// Row-major bf16 matrix [rows, inner] -> tensor map with 64 x 128 boxes,
// 128-byte swizzle, zero fill outside the matrix.
int make_tmap(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return MOE_ECUDA;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {BK, BN_HALF};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
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

template <bool SWIGLU>
int smem_attr_once(int device) {
  static std::mutex mu;
  static bool done[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return MOE_ECUDA;
  if (!done[device]) {
    if (cudaFuncSetAttribute(grouped_gemm_tc_kernel<SWIGLU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES)) != cudaSuccess) {
      return MOE_ECUDA;
    }
    done[device] = true;
  }
  return MOE_OK;
}

template <bool SWIGLU>
int launch_gemm(const void* A, const void* B0, const void* B1, const int32_t* offsets, void* out, int Tk, int K,
                int n_out, int b_rows, int E, const Ctx& c, cudaStream_t s) {
  if (Tk <= 0) return MOE_OK;
  CUtensorMap ta, tb0, tb1;
  int rc = make_tmap(&ta, A, static_cast<uint64_t>(K), static_cast<uint64_t>(Tk));
  if (rc != MOE_OK) return rc;
  rc = make_tmap(&tb0, B0, static_cast<uint64_t>(K), static_cast<uint64_t>(E) * b_rows);
  if (rc != MOE_OK) return rc;
  if (SWIGLU) {
    rc = make_tmap(&tb1, B1, static_cast<uint64_t>(K), static_cast<uint64_t>(E) * b_rows);
    if (rc != MOE_OK) return rc;
  } else {
    tb1 = tb0;
  }
  rc = smem_attr_once<SWIGLU>(c.device);
  if (rc != MOE_OK) return rc;
  GemmArgs a;
  a.offsets = offsets;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.ldo = n_out;
  a.n_out = n_out;
  a.b_rows = b_rows;
  a.K = K;
  a.Tk = Tk;
  a.E = E;
  a.n_tiles = SWIGLU ? (n_out + BN_HALF - 1) / BN_HALF : (n_out + BN - 1) / BN;
  a.status = c.status;
  a.wait_ns = c.wait_ns;
  // Upper bound on tiles: whole row blocks plus at most one partial block
  // per expert that has rows (at most min(E, Tk) of them).
  const long long max_tiles = (static_cast<long long>(Tk) / BM + (E < Tk ? E : Tk)) * a.n_tiles;
  const int grid = balanced_grid(max_tiles, c.num_sms);
  launch_pdl(grouped_gemm_tc_kernel<SWIGLU>, grid, NUM_THREADS, SMEM_BYTES, s, ta, tb0, tb1, a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ECUDA;
}

}  // namespace

int launch_tc_gate_up(const void* x_perm, const int32_t* offsets, const void* W1, const void* W3, void* h, int Tk,
                      int d, int dff, int E, const Ctx& c, cudaStream_t s) {
  return launch_gemm<true>(x_perm, W1, W3, offsets, h, Tk, d, dff, dff, E, c, s);
}

int launch_tc_down(const void* h, const int32_t* offsets, const void* W2, void* y, int Tk, int d, int dff, int E,
                   const Ctx& c, cudaStream_t s) {
  return launch_gemm<false>(h, W2, nullptr, offsets, y, Tk, dff, d, d, E, c, s);
}

}  // namespace moe
