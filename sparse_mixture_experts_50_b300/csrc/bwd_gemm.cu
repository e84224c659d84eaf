// Backward of the expert GEMMs (Mixtral 8x7B model reference page, Training:
// the experts and the router are trained together; "The Evolving
// Transformer - 05 Mixtral", section 04, SwiGLU: y = W2 (silu(W1 x) * W3 x)).
// For the rows p of expert e, with dout gathered per routed row and w_p the
// row's gate weight:
//   dh = w_p (dout W2_e)                                           (DH, fp32)
//   a = x W1_e^T,  b = x W3_e^T,
//   da = dh * b * silu'(a),  db = dh * silu(a)                     (DSW)
//   When the forward kept p = b silu'(a) and q = silu(a) (bf16, formed from
//   its fp32 a and b), DH's epilogue forms da = dh p and db = dh q from its
//   fp32 dh directly and DSW does not run.
//   dx_perm = da W1_e + db W3_e                                    (DX)
//   dW2_e = dy^T h,  dW1_e = da^T x,  dW3_e = db^T x               (WGRAD)
//
// One persistent tcgen05 kernel template, one CTA per SM, warp-specialised
// like the forward kernel (warp 0 TMA, warp 1 MMA + tensor memory, warps 2-5
// epilogue), every operand staged by TMA with the 128-byte swizzle.  The
// token rows of DH, DSW and DX are K-major; everything else is read in place
// MN-major, as TMA boxes of 64 M or N columns x 64 K rows described to
// tcgen05 with the transpose bits: the weights of DH and DX (W2 [E,d,F] for
// dh, W1 and W3 [E,F,d] for dx_perm, whose contiguous dimension is the
// GEMM's N) and both operands of WGRAD (the token-major activations
// [Tk, channels], K = the expert's tokens).  An expert's last K block of
// WGRAD may run into the next expert's rows: the MMA warp clears those rows
// (up to the next 16-row MMA step) in shared memory and skips the steps
// past them.
//   DH       tile 128 rows x 256 h columns, one K=d pass; the epilogue
//            scales by w_p and stores fp32 (dout is gathered exactly and dh
//            stays fp32: a bf16 rounding of w dout or of dh would be
//            amplified by the 4096-term sum where it cancels), or, given
//            the kept p and q, reads them (one 32-column chunk ahead) and
//            stores da, db in bf16.
//   DSW      tile 128 rows x 128 h columns: a and b recomputed in one K=d
//            pass over the W1 and W3 rows (N=256, as the forward's gate/up
//            GEMM); the epilogue reads dh, forms da, db in fp32 and rounds
//            them to bf16.
//   DX       tile 128 rows x 256 columns of dx_perm; two K=F passes (da with
//            W1, then db with W3) into one accumulator; two accumulators
//            alternate between tiles.
//   WGRAD    per expert an [M, N] fp32 matrix, tile 128 x 256, K = the
//            expert's routed rows; an expert with no tokens gets zeros (its
//            tiles skip the MMAs).
// Epilogue stores go through a per-warp 32 x 32 staging block in shared
// memory, so that each store instruction writes contiguous row segments
// (a lane per row would make every instruction touch 32 rows).
// Every wait is bounded as in the forward kernel.
#include <cuda.h>
#include <mutex>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

enum { MODE_DH = 0, MODE_DX = 1, MODE_WGRAD = 2, MODE_DSW = 3 };

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BNH = 128;                  // one B box
constexpr int UMMA_K = 16;
constexpr int A_BYTES = BM * BK * 2;      // 16 KB
constexpr int B_BYTES = 2 * BNH * BK * 2; // up to two B boxes, 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int STAGES = 4;
constexpr int THREADS = 192;
constexpr int EPI_THREADS = 128;
constexpr int MAX_E = 64;
constexpr int MN_BOX_BYTES = 64 * BK * 2; // one MN-major box: 64 columns x 64 K rows

struct Ctl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int tile_prefix[MAX_E + 1];
  int mtiles[MAX_E];
  int seg[MAX_E + 1];    // routed-row segments
  int rows[MAX_E];       // WGRAD: tokens of each expert
};

constexpr int STG_PITCH = 33;             // staging block row pitch (32-bit words)
constexpr int STG_WORDS = 32 * STG_PITCH;  // one warp's staging block
constexpr size_t CTL_BYTES = (sizeof(Ctl) + 15) / 16 * 16;
constexpr int KEEP_WORDS = 2 * 32 * 16;    // DH: one warp's p and q chunk (32 rows x 32 bf16 each)
constexpr size_t SMEM_BYTES = 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + CTL_BYTES +
                              4 * STG_WORDS * sizeof(uint32_t) + 4 * KEEP_WORDS * sizeof(uint32_t);
static_assert(SMEM_BYTES <= 232448, "shared memory per block");

struct BwdArgs {
  const int32_t* offsets;  // [E+1] routed-row boundaries
  int b_krows;             // DH, DX: K rows per expert in the MN-major weight (d, F)
  int E;
  int Tk;
  int K;                   // reduction length of one pass (d, F; WGRAD: unused)
  int b_rows;              // rows per expert in the B tensor(s)
  int n_out;               // output columns (DH, DSW: F; DX: d; WGRAD: N)
  int m_rows;              // WGRAD: output rows M
  int n_tiles;
  // DSW: out0 = dA, out1 = dB [Tk, F]; DX: out0 = dx_perm [Tk, d]
  __nv_bfloat16* out0;
  __nv_bfloat16* out1;
  float* outf;             // WGRAD: [E, M, N]; DH: dh [Tk, F]
  const float* w_perm;     // DH: gate weight of each routed row [Tk]
  const float* dh;         // DSW: dh [Tk, F] fp32
  const __nv_bfloat16* keep;  // DH, optional: the forward's p, q planes [2, Tk, F]
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

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// The helpers below unroll their 32 rows fully (rows past `rows` are
// predicated off), so that a warp has all its loads or stores in flight at
// once instead of one row's latency after another.

// The warp's 32 rows x 32 fp32 columns (lane = row, v[i] = column i) to
// dst[r * ld + i] for r < rows.  Each lane writes its row into the staging
// block as eight 16-byte units (unit j of row r at unit j ^ (r & 7), so the
// eight lanes of a quarter-warp meet distinct banks); then every load/store
// instruction moves four whole 128-byte rows, a quarter-warp per row.
__device__ __forceinline__ void warp_store_f32(uint32_t* stg, const uint32_t (&v)[32], float* dst, size_t ld,
                                               int rows, int lane) {
  const uint32_t base = ptx::smem_u32(stg);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    ptx::sts128(base + lane * 128 + ((j ^ (lane & 7)) << 4),
                make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
  __syncwarp();
  const int sub = lane >> 3, u = lane & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 4 * i + sub;
    const uint4 val = ptx::lds128(base + r * 128 + ((u ^ (r & 7)) << 4));
    if (r < rows) *reinterpret_cast<uint4*>(dst + r * ld + 4 * u) = val;
  }
  __syncwarp();
}

// Rows r < rows of src (row stride ld, 32 fp32 each; lane = column), one
// 128-byte row per instruction; rows past `rows` read as zero.
__device__ __forceinline__ void warp_load_rows_f32(const float* src, size_t ld, int rows, int lane, float (&t)[32]) {
#pragma unroll
  for (int r = 0; r < 32; ++r) t[r] = r < rows ? __ldg(src + r * ld + lane) : 0.0f;
}

// The transpose of what warp_load_rows_f32 read: lane = row, v[i] = column i.
__device__ __forceinline__ void warp_transpose_f32(uint32_t* stg, const float (&t)[32], int lane, float (&v)[32]) {
#pragma unroll
  for (int r = 0; r < 32; ++r) stg[r * STG_PITCH + lane] = __float_as_uint(t[r]);
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(stg[lane * STG_PITCH + i]);
  __syncwarp();
}

// The SwiGLU derivative for h = silu(a) b, given dh = g:
// da = g b silu'(a) with silu'(a) = s (1 + a (1 - s)), s = sigmoid(a); db = g silu(a).
__device__ __forceinline__ void swiglu_grad(float g, float a, float b, float& da, float& db) {
  const float s = __frcp_rn(1.0f + __expf(-a));  // = 1.0f / (1 + e^-a), correctly rounded
  da = g * b * (s * (1.0f + a * (1.0f - s)));
  db = g * (a * s);
}

// The warp's 32 rows x 32 bf16 columns (lane = row, pk[i] = columns 2i,
// 2i+1) to dst[r * ld + ...] for r < rows.  Each lane writes its 64-byte row
// as four 16-byte units (unit j of row r at unit j ^ ((r >> 1) & 3), so a
// quarter-warp meets distinct banks); then every load/store instruction moves
// eight whole rows, four lanes per row.
__device__ __forceinline__ void warp_store_bf16(uint32_t* stg, const uint32_t (&pk)[16], __nv_bfloat16* dst,
                                                size_t ld, int rows, int lane) {
  const uint32_t base = ptx::smem_u32(stg);
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    ptx::sts128(base + lane * 64 + ((j ^ sw) << 4), make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]));
  __syncwarp();
  const int sub = lane >> 2, u = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 8 * i + sub;
    const uint4 val = ptx::lds128(base + r * 64 + ((u ^ ((r >> 1) & 3)) << 4));
    if (r < rows) *reinterpret_cast<uint4*>(dst + r * ld + 8 * u) = val;
  }
  __syncwarp();
}

template <int MODE>
struct Shape {
  static constexpr int passes = MODE == MODE_DX ? 2 : 1;
  static constexpr int n_tile = MODE == MODE_DSW ? BNH : 2 * BNH;   // output columns per tile
  static constexpr int acc_cols = 2 * BNH;
  static constexpr int n_acc = 2;                                    // accumulators in flight
  static constexpr int tmem_cols = 512;
  static constexpr bool a_mn = MODE == MODE_WGRAD;                               // activations MN-major
  static constexpr bool b_mn = MODE == MODE_DH || MODE == MODE_DX || MODE == MODE_WGRAD;
  static constexpr uint32_t idesc = a_mn   ? ptx::idesc_bf16_f32_mn(BM, 2 * BNH)
                                    : b_mn ? ptx::idesc_bf16_f32_bmn(BM, 2 * BNH)
                                           : ptx::idesc_bf16_f32(BM, 2 * BNH);
};

// Tensor maps per pass: A (token rows or, WGRAD, channel rows) and B.
struct Maps {
  CUtensorMap a[3];
  CUtensorMap b[3];
};

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1) bwd_gemm_kernel(const __grid_constant__ Maps maps, const BwdArgs args) {
  using S = Shape<MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + STAGES * STAGE_BYTES);
  uint32_t* stage_blocks = reinterpret_cast<uint32_t*>(smem + STAGES * STAGE_BYTES + CTL_BYTES);
  uint32_t* keep_blocks = stage_blocks + 4 * STG_WORDS;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const volatile int* abort_flag = &ctl->abort_flag;

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
    for (int p = 0; p < 3; ++p) {
      ptx::prefetch_tmap(&maps.a[p]);
      ptx::prefetch_tmap(&maps.b[p]);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(&ctl->tmem_base, S::tmem_cols);
    ptx::tmem_relinquish();
  }
  pdl_enter();
  if (threadIdx.x == 0) {
    int prev = 0;
    int run = 0;
    ctl->tile_prefix[0] = 0;
    for (int e = 0; e <= args.E; ++e) {
      int o = args.offsets[e];
      if (o < prev || o > args.Tk) {
        record_status(args.status, MOE_EDEVICE);
        o = prev;
      }
      if (e > 0) {
        const int n_e = o - prev;
        ctl->seg[e - 1] = prev;
        if (MODE == MODE_WGRAD) {
          ctl->rows[e - 1] = n_e;
          const int mt = (args.m_rows + BM - 1) / BM;
          ctl->mtiles[e - 1] = mt;
          run += mt * args.n_tiles;
        } else {
          const int mt = (n_e + BM - 1) / BM;
          ctl->mtiles[e - 1] = mt;
          run += mt * args.n_tiles;
        }
        ctl->tile_prefix[e] = run;
      }
      prev = o;
    }
    ctl->seg[args.E] = prev;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  const int total_tiles = ctl->tile_prefix[args.E];
  const int kb_pass = (args.K + BK - 1) / BK;

  // K steps of a tile (all passes).
  auto tile_kblocks = [&](int e) -> int {
    if (MODE == MODE_WGRAD) return (ctl->rows[e] + BK - 1) / BK;
    return S::passes * kb_pass;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t filled = 0;
      uint32_t last_parity[STAGES];
      for (int s = 0; s < STAGES; ++s) last_parity[s] = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        int e, m, n;
        decode_tile(ctl, args.E, tile, e, m, n);
        const int nkb = tile_kblocks(e);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!ptx::mbar_wait(&ctl->empty[stage], phase ^ 1u, abort_flag, args.wait_ns)) {
            raise_abort(ctl, args.status);
            ok = false;
            break;
          }
          const int pass = MODE == MODE_WGRAD ? 0 : kb / kb_pass;
          const int kx = (kb - pass * kb_pass) * BK;
          const int arow = ctl->seg[e] + m * BM;
          const int brow = e * args.b_rows + n * S::n_tile;
          uint8_t* sa = smem + stage * STAGE_BYTES;
          ptx::mbar_arrive_expect_tx(&ctl->full[stage], STAGE_BYTES);
          if (MODE == MODE_WGRAD) {
            // Two 64-channel boxes of A and four of B, K rows = the
            // expert's tokens seg[e] + kb*64 .. +63.
            const int krow = ctl->seg[e] + kb * BK;
#pragma unroll
            for (int i = 0; i < 2; ++i)
              ptx::tma_load_2d(sa + i * MN_BOX_BYTES, &maps.a[0], &ctl->full[stage], m * BM + 64 * i, krow);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              ptx::tma_load_2d(sa + A_BYTES + i * MN_BOX_BYTES, &maps.b[0], &ctl->full[stage],
                               n * 2 * BNH + 64 * i, krow);
          } else if (S::b_mn) {
            ptx::tma_load_2d(sa, &maps.a[pass], &ctl->full[stage], kx, arow);
            // Four 64-column x 64-row boxes: N columns n*256 + 64i, K rows
            // kx .. kx+63 of expert e.
            const int krow = e * args.b_krows + kx;
#pragma unroll
            for (int i = 0; i < 4; ++i)
              ptx::tma_load_2d(sa + A_BYTES + i * MN_BOX_BYTES, &maps.b[pass], &ctl->full[stage],
                               n * S::n_tile + 64 * i, krow);
          } else {
            ptx::tma_load_2d(sa, &maps.a[pass], &ctl->full[stage], kx, arow);
            // DSW stages the W1 and the W3 rows of its 128 h columns; WGRAD
            // two consecutive 128-row boxes of one tensor.
            ptx::tma_load_2d(sa + A_BYTES, &maps.b[pass], &ctl->full[stage], kx, brow);
            if (MODE == MODE_DSW)
              ptx::tma_load_2d(sa + A_BYTES + BNH * BK * 2, &maps.b[1], &ctl->full[stage], kx, brow);
            else
              ptx::tma_load_2d(sa + A_BYTES + BNH * BK * 2, &maps.b[pass], &ctl->full[stage], kx, brow + BNH);
          }
          filled |= 1u << stage;
          last_parity[stage] = phase;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < STAGES; ++s) {
        if (filled & (1u << s)) ptx::mbar_wait(&ctl->full[s], last_parity[s], nullptr, drain_limit(args.wait_ns));
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------- MMA issuer
    // Lane 0 waits and issues; the whole warp clears WGRAD's ragged rows.
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
      int e, m, n;
      decode_tile(ctl, args.E, tile, e, m, n);
      const int nkb = tile_kblocks(e);
      bool got = true;
      if (lane == 0) {
        got = ptx::mbar_wait(&ctl->tempty[acc], acc_phase ^ 1u, abort_flag, args.wait_ns);
        if (!got) raise_abort(ctl, args.status);
      }
      if (!__shfl_sync(0xFFFFFFFFu, got, 0)) break;
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * S::acc_cols);
      for (int kb = 0; kb < nkb; ++kb) {
        if (lane == 0) {
          got = ptx::mbar_wait(&ctl->full[stage], phase, abort_flag, args.wait_ns);
          if (!got) raise_abort(ctl, args.status);
        }
        if (!__shfl_sync(0xFFFFFFFFu, got, 0)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        // Every pass adds into the same accumulator (DX: da W1 + db W3).
        const int pass = MODE == MODE_WGRAD ? 0 : kb / kb_pass;
        const int kin = MODE == MODE_WGRAD ? kb : kb - pass * kb_pass;
        const bool first = MODE == MODE_DX ? (kb == 0) : (kin == 0);
        const uint32_t sa = ptx::smem_u32(smem + stage * STAGE_BYTES);
        const uint32_t sb = sa + A_BYTES;
        int ksteps = BK / UMMA_K;
        if (MODE == MODE_WGRAD) {
          const int valid = ctl->rows[e] - kb * BK;  // >= 1
          if (valid < BK) {
            const int upto = (valid + UMMA_K - 1) / UMMA_K * UMMA_K;
            ksteps = upto / UMMA_K;
            // Rows valid .. upto-1 of the six boxes (A: 2, B: 4) hold the
            // next expert's tokens: zero them.  A 128-byte row keeps its
            // bytes under the swizzle, which only permutes its 16-byte chunks.
            const int per_box = (upto - valid) * 8;
            const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
            for (int i = lane; i < 6 * per_box; i += 32) {
              const int box = i / per_box;
              const int rem = i - box * per_box;
              ptx::sts128(sa + box * MN_BOX_BYTES + (valid + (rem >> 3)) * 128 + (rem & 7) * 16, zero);
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
          }
        }
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            if (kk < ksteps) {
              // MN-major operands: a K step of 16 is two 8-row groups, 2048 bytes on.
              const uint64_t adesc = S::a_mn ? ptx::sdesc_mnmajor_sw128(sa + kk * 2048, MN_BOX_BYTES)
                                             : ptx::sdesc_kmajor_sw128(sa + kk * UMMA_K * 2);
              const uint64_t bdesc = S::b_mn ? ptx::sdesc_mnmajor_sw128(sb + kk * 2048, MN_BOX_BYTES)
                                             : ptx::sdesc_kmajor_sw128(sb + kk * UMMA_K * 2);
              ptx::umma_bf16(d_tmem, adesc, bdesc, S::idesc, (first && kk == 0) ? 0u : 1u);
            }
          }
          ptx::umma_commit(&ctl->empty[stage]);
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) {
        if (nkb > 0) {
          ptx::umma_commit(&ctl->tfull[acc]);
        } else {
          ptx::mbar_arrive(&ctl->tfull[acc]);  // nothing to wait for: the epilogue writes zeros
        }
      }
      __syncwarp();
      if (++acc == S::n_acc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) {
      ptx::umma_commit(&ctl->drain);
      ptx::mbar_wait(&ctl->drain, 0, nullptr, drain_limit(args.wait_ns));
    }
  } else {
    // -------------------------------------------------- epilogue (warps 2-5)
    const int quad = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    // DH with the kept p and q: each lane asks L2 for its row of a tile's p
    // and q one tile ahead, so that the epilogue's loads hit L2.
    auto prefetch_keep = [&](int t) {
      if (MODE != MODE_DH || args.keep == nullptr || t >= total_tiles) return;
      int pe, pm, pn;
      decode_tile(ctl, args.E, t, pe, pm, pn);
      const int prow0 = ctl->seg[pe] + pm * BM + quad * 32;
      const int prows = max(0, min(32, ctl->seg[pe + 1] - prow0));
      const int pcol0 = pn * 2 * BNH;
      const int ncols = min(2 * BNH, args.n_out - pcol0);
      if (lane < prows && ncols > 0) {
        const size_t o = static_cast<size_t>(prow0 + lane) * args.n_out + pcol0;
        ptx::prefetch_l2_bulk(args.keep + o, static_cast<uint32_t>(ncols) * 2u);
        ptx::prefetch_l2_bulk(args.keep + static_cast<size_t>(args.Tk) * args.n_out + o,
                              static_cast<uint32_t>(ncols) * 2u);
      }
    };
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      int e, m, n;
      decode_tile(ctl, args.E, tile, e, m, n);
      if (tile == blockIdx.x) prefetch_keep(tile);
      prefetch_keep(tile + gridDim.x);
      const bool ready = ptx::mbar_wait(&ctl->tfull[acc], acc_phase, abort_flag, args.wait_ns);
      if (!__all_sync(0xFFFFFFFFu, ready)) {
        raise_abort(ctl, args.status);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t t_row =
          tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * S::acc_cols);
      uint32_t* stg = stage_blocks + quad * STG_WORDS;
      if (MODE == MODE_DH) {
        const int row0 = ctl->seg[e] + m * BM + quad * 32;  // the warp's first row
        const int rows = max(0, min(32, ctl->seg[e + 1] - row0));
        const int col0 = n * 2 * BNH;
        const float wp = lane < rows ? __ldg(args.w_perm + row0 + lane) : 0.0f;
        if (args.keep != nullptr) {
          // dh stays in registers: da = dh p, db = dh q.  The p and q rows of
          // the next 32-column chunk are copied asynchronously into the
          // warp's keep block while this chunk is worked on; word w of row r
          // sits at r*16 + (w ^ (r & 15)), so the transposed reads (lane =
          // row) meet at most two lanes per bank.
          uint32_t* kb = keep_blocks + quad * KEEP_WORDS;
          const uint32_t kb_s = ptx::smem_u32(kb);
          const __nv_bfloat16* qplane = args.keep + static_cast<size_t>(args.Tk) * args.n_out;
          const size_t rbase = static_cast<size_t>(row0) * args.n_out + col0;
          const int half = lane >> 4, w = lane & 15;
          auto issue = [&](int c) {
            const int lr = (rows > 0 && col0 + c < args.n_out) ? rows : 0;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int r = 2 * i + half;
              const bool ok = r < lr;
              const size_t off = ok ? rbase + static_cast<size_t>(r) * args.n_out + c + 2 * w : 0;
              const uint32_t dst = kb_s + static_cast<uint32_t>(r * 16 + (w ^ (r & 15))) * 4u;
              ptx::cp_async_4(dst, args.keep + off, ok ? 4u : 0u);
              ptx::cp_async_4(dst + 32 * 16 * 4, qplane + off, ok ? 4u : 0u);
            }
            ptx::cp_async_commit();
          };
          issue(0);
#pragma unroll 1
          for (int c = 0; c < 2 * BNH; c += 32) {
            const bool live = rows > 0 && col0 + c < args.n_out;
            ptx::cp_async_wait_all();
            __syncwarp();
            uint32_t pa[16], pb[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              pa[i] = kb[lane * 16 + (i ^ (lane & 15))];
              pb[i] = kb[32 * 16 + lane * 16 + (i ^ (lane & 15))];
            }
            __syncwarp();
            if (c + 32 < 2 * BNH) issue(c + 32);
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(t_row + c, v);
            ptx::tmem_ld_wait();
            if (live) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float2 p2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pa[i]));
                const float2 q2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pb[i]));
                const float g0 = wp * __uint_as_float(v[2 * i]);
                const float g1 = wp * __uint_as_float(v[2 * i + 1]);
                pa[i] = pack_bf16x2(g0 * p2.x, g1 * p2.y);
                pb[i] = pack_bf16x2(g0 * q2.x, g1 * q2.y);
              }
              warp_store_bf16(stg, pa, args.out0 + rbase + c, args.n_out, rows, lane);
              warp_store_bf16(stg, pb, args.out1 + rbase + c, args.n_out, rows, lane);
            }
          }
        } else {
#pragma unroll 1
        for (int c = 0; c < 2 * BNH; c += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(t_row + c, v);
          ptx::tmem_ld_wait();
          if (rows > 0 && col0 + c < args.n_out) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(wp * __uint_as_float(v[i]));
            warp_store_f32(stg, v, args.outf + static_cast<size_t>(row0) * args.n_out + col0 + c, args.n_out, rows,
                           lane);
          }
        }
        }
      } else if (MODE == MODE_DSW) {
        const int row0 = ctl->seg[e] + m * BM + quad * 32;
        const int rows = max(0, min(32, ctl->seg[e + 1] - row0));
        const int col0 = n * BNH;
#pragma unroll 1
        for (int c = 0; c < BNH; c += 32) {
          const bool live = rows > 0 && col0 + c < args.n_out;
          const size_t base = static_cast<size_t>(row0) * args.n_out + col0 + c;
          // dh's loads go out before the accumulator is read.
          float t[32];
          warp_load_rows_f32(args.dh + base, args.n_out, live ? rows : 0, lane, t);
          uint32_t av[32], bv[32];
          ptx::tmem_ld_32x32b_x32(t_row + c, av);
          ptx::tmem_ld_32x32b_x32(t_row + BNH + c, bv);
          ptx::tmem_ld_wait();
          if (live) {
            float g[32];
            warp_transpose_f32(stg, t, lane, g);
            uint32_t pa[16], pb[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float da[2], db[2];
#pragma unroll
              for (int h = 0; h < 2; ++h)
                swiglu_grad(g[2 * i + h], __uint_as_float(av[2 * i + h]), __uint_as_float(bv[2 * i + h]), da[h], db[h]);
              pa[i] = pack_bf16x2(da[0], da[1]);
              pb[i] = pack_bf16x2(db[0], db[1]);
            }
            warp_store_bf16(stg, pa, args.out0 + base, args.n_out, rows, lane);
            warp_store_bf16(stg, pb, args.out1 + base, args.n_out, rows, lane);
          }
        }
      } else if (MODE == MODE_DX) {
        const int row0 = ctl->seg[e] + m * BM + quad * 32;
        const int rows = max(0, min(32, ctl->seg[e + 1] - row0));
        const int col0 = n * 2 * BNH;
#pragma unroll 1
        for (int c = 0; c < 2 * BNH; c += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(t_row + c, v);
          ptx::tmem_ld_wait();
          if (rows > 0 && col0 + c < args.n_out) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
            warp_store_bf16(stg, pk, args.out0 + static_cast<size_t>(row0) * args.n_out + col0 + c, args.n_out, rows,
                            lane);
          }
        }
      } else {
        // WGRAD: rows m*128 + quad*32 .. of expert e's [M, N] fp32 gradient.
        const int row0 = m * BM + quad * 32;
        const int rows = max(0, min(32, args.m_rows - row0));
        const bool empty = ctl->rows[e] == 0;
        const int col0 = n * 2 * BNH;
        float* base = args.outf + (static_cast<size_t>(e) * args.m_rows + row0) * args.n_out;
#pragma unroll 1
        for (int c = 0; c < 2 * BNH; c += 32) {
          uint32_t v[32];
          if (!empty) {
            ptx::tmem_ld_32x32b_x32(t_row + c, v);
            ptx::tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
          }
          if (rows > 0 && col0 + c < args.n_out) warp_store_f32(stg, v, base + col0 + c, args.n_out, rows, lane);
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&ctl->tempty[acc]);
      if (++acc == S::n_acc) {
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
    ptx::tmem_dealloc(tmem_base, S::tmem_cols);
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

// Row-major bf16 [rows, inner] -> 64 x box_rows boxes, 128-byte swizzle, zero fill.
int make_tmap(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, int box_rows = BNH) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return MOE_ECUDA;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {BK, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ECUDA;
}

template <int MODE>
int smem_attr_once(int device) {
  static std::mutex mu;
  static bool done[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return MOE_ECUDA;
  if (!done[device]) {
    if (cudaFuncSetAttribute(bwd_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES)) != cudaSuccess)
      return MOE_ECUDA;
    done[device] = true;
  }
  return MOE_OK;
}

template <int MODE>
int launch_bwd(const Maps& maps, BwdArgs a, long long max_tiles, const Ctx& c, cudaStream_t s) {
  int rc = smem_attr_once<MODE>(c.device);
  if (rc != MOE_OK) return rc;
  a.status = c.status;
  a.wait_ns = c.wait_ns;
  long long grid = max_tiles < c.num_sms ? max_tiles : c.num_sms;
  if (grid < 1) grid = 1;
  launch_pdl(bwd_gemm_kernel<MODE>, static_cast<int>(grid), THREADS, SMEM_BYTES, s, maps, a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ECUDA;
}

}  // namespace

int launch_bwd_dh(const void* dout_perm, const float* w_perm, const int32_t* offsets, const void* W2, float* dh,
                  const void* keep, void* dA, void* dB, int Tk, int d, int dff, int E, const Ctx& c,
                  cudaStream_t s) {
  if (Tk <= 0) return MOE_OK;
  Maps m;
  int rc = make_tmap(&m.a[0], dout_perm, d, Tk);
  if (rc == MOE_OK) rc = make_tmap(&m.b[0], W2, dff, static_cast<uint64_t>(E) * d, 64);  // MN-major: [E*d, F]
  if (rc != MOE_OK) return rc;
  m.a[1] = m.a[2] = m.a[0];
  m.b[1] = m.b[2] = m.b[0];
  BwdArgs a = {};
  a.offsets = offsets;
  a.E = E;
  a.Tk = Tk;
  a.K = d;
  a.b_rows = dff;
  a.b_krows = d;
  a.n_out = dff;
  a.n_tiles = (dff + 2 * BNH - 1) / (2 * BNH);
  a.outf = dh;
  a.w_perm = w_perm;
  a.keep = static_cast<const __nv_bfloat16*>(keep);
  a.out0 = static_cast<__nv_bfloat16*>(dA);
  a.out1 = static_cast<__nv_bfloat16*>(dB);
  const long long max_tiles = (static_cast<long long>(Tk) / BM + (E < Tk ? E : Tk)) * a.n_tiles;
  return launch_bwd<MODE_DH>(m, a, max_tiles, c, s);
}

int launch_bwd_dsw(const void* x_perm, const float* dh, const int32_t* offsets, const void* W1, const void* W3,
                   void* dA, void* dB, int Tk, int d, int dff, int E, const Ctx& c, cudaStream_t s) {
  if (Tk <= 0) return MOE_OK;
  Maps m;
  int rc = make_tmap(&m.a[0], x_perm, d, Tk);
  if (rc == MOE_OK) rc = make_tmap(&m.b[0], W1, d, static_cast<uint64_t>(E) * dff);
  if (rc == MOE_OK) rc = make_tmap(&m.b[1], W3, d, static_cast<uint64_t>(E) * dff);
  if (rc != MOE_OK) return rc;
  m.a[1] = m.a[2] = m.a[0];
  m.b[2] = m.b[1];
  BwdArgs a = {};
  a.offsets = offsets;
  a.E = E;
  a.Tk = Tk;
  a.K = d;
  a.b_rows = dff;
  a.n_out = dff;
  a.n_tiles = (dff + BNH - 1) / BNH;
  a.out0 = static_cast<__nv_bfloat16*>(dA);
  a.out1 = static_cast<__nv_bfloat16*>(dB);
  a.dh = dh;
  const long long max_tiles = (static_cast<long long>(Tk) / BM + (E < Tk ? E : Tk)) * a.n_tiles;
  return launch_bwd<MODE_DSW>(m, a, max_tiles, c, s);
}

int launch_bwd_dx(const void* dA, const void* dB, const int32_t* offsets, const void* W1, const void* W3,
                  void* dx_perm, int Tk, int d, int dff, int E, const Ctx& c, cudaStream_t s) {
  if (Tk <= 0) return MOE_OK;
  Maps m;
  int rc = make_tmap(&m.a[0], dA, dff, Tk);
  if (rc == MOE_OK) rc = make_tmap(&m.a[1], dB, dff, Tk);
  if (rc == MOE_OK) rc = make_tmap(&m.b[0], W1, d, static_cast<uint64_t>(E) * dff, 64);  // MN-major: [E*F, d]
  if (rc == MOE_OK) rc = make_tmap(&m.b[1], W3, d, static_cast<uint64_t>(E) * dff, 64);
  if (rc != MOE_OK) return rc;
  m.a[2] = m.a[1];
  m.b[2] = m.b[1];
  BwdArgs a = {};
  a.offsets = offsets;
  a.E = E;
  a.Tk = Tk;
  a.K = dff;
  a.b_rows = d;
  a.b_krows = dff;
  a.n_out = d;
  a.n_tiles = (d + 2 * BNH - 1) / (2 * BNH);
  a.out0 = static_cast<__nv_bfloat16*>(dx_perm);
  const long long max_tiles = (static_cast<long long>(Tk) / BM + (E < Tk ? E : Tk)) * a.n_tiles;
  return launch_bwd<MODE_DX>(m, a, max_tiles, c, s);
}

int launch_bwd_wgrad(const void* A, const void* B, const int32_t* offsets, float* dW, int M, int N, int Tk, int E,
                     const Ctx& c, cudaStream_t s) {
  Maps m;
  // Token-major [Tk, M] and [Tk, N], read MN-major (64 x 64 boxes).
  const uint64_t rows = static_cast<uint64_t>(Tk > 0 ? Tk : 1);
  int rc = make_tmap(&m.a[0], A, static_cast<uint64_t>(M), rows, 64);
  if (rc == MOE_OK) rc = make_tmap(&m.b[0], B, static_cast<uint64_t>(N), rows, 64);
  if (rc != MOE_OK) return rc;
  m.a[1] = m.a[2] = m.a[0];
  m.b[1] = m.b[2] = m.b[0];
  BwdArgs a = {};
  a.offsets = offsets;
  a.E = E;
  a.Tk = Tk;
  a.K = 0;
  a.b_rows = 0;
  a.n_out = N;
  a.m_rows = M;
  a.n_tiles = (N + 2 * BNH - 1) / (2 * BNH);
  a.outf = dW;
  const long long max_tiles = static_cast<long long>(E) * ((M + BM - 1) / BM) * a.n_tiles;
  return launch_bwd<MODE_WGRAD>(m, a, max_tiles, c, s);
}

}  // namespace moe
