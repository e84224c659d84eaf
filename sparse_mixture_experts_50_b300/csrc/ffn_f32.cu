// Steps a4-a5 in fp32 on the CUDA cores (no TF32): the grouped expert GEMMs
// of the sparse-MoE layer for fp32 storage ("The Evolving Transformer - 05
// Mixtral", section 04 SwiGLU: down(silu(gate x) * up x)).
//
// One CTA computes a 64x64 output tile of one expert's row segment: 256
// threads, 4x4 outputs each, K staged through shared memory 16 at a time.
// The gate/up kernel keeps two accumulators (W1 and W3 rows of the same
// output column) and writes h = silu(a) * b; the down kernel writes y.
// The CTA's expert and row block come from the device-side offsets[E+1],
// so the host never reads the per-expert counts.
#include <math.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, kThreads = 256;

// Finds the expert and first row of row-block `mt` (blocks of BM rows,
// numbered expert by expert).  Returns false if there is no such block.
__device__ __forceinline__ bool find_block(const int32_t* offsets, int E, int Tk, int mt, int& e_out, int& row0,
                                           int& row_end) {
  int acc = 0;
  for (int e = 0; e < E; ++e) {
    const int beg = offsets[e];
    const int end = min(offsets[e + 1], Tk);
    const int n = end - beg;
    const int blocks = n > 0 ? (n + BM - 1) / BM : 0;
    if (mt < acc + blocks) {
      e_out = e;
      row0 = beg + (mt - acc) * BM;
      row_end = end;
      return true;
    }
    acc += blocks;
  }
  return false;
}

template <bool SWIGLU>
__global__ void __launch_bounds__(kThreads) ffn_f32_kernel(const float* __restrict__ A, const int32_t* __restrict__ offsets,
                                                           const float* __restrict__ B0, const float* __restrict__ B1,
                                                           float* __restrict__ out, int Tk, int E, int K, int N,
                                                           int b_rows) {
  pdl_enter();
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs0[BK][BN + 4];
  __shared__ float Bs1[BK][BN + 4];  // W3 tile (gate/up kernel only)
  int e, row0, row_end;
  if (!find_block(offsets, E, Tk, blockIdx.y, e, row0, row_end)) return;
  const int n0 = blockIdx.x * BN;
  const int tid = threadIdx.x;
  const int ty = tid / 16, tx = tid % 16;  // 16 x 16 threads, 4 x 4 outputs each
  float acc0[4][4] = {}, acc1[4][4] = {};
  const float* b0 = B0 + static_cast<size_t>(e) * b_rows * K;
  const float* b1 = SWIGLU ? B1 + static_cast<size_t>(e) * b_rows * K : nullptr;
  for (int k0 = 0; k0 < K; k0 += BK) {
    for (int i = tid; i < BM * BK; i += kThreads) {
      const int r = i / BK, kk = i % BK;
      const int gr = row0 + r, gk = k0 + kk;
      As[kk][r] = (gr < row_end && gk < K) ? A[static_cast<size_t>(gr) * K + gk] : 0.0f;
      const int br = n0 + r;
      Bs0[kk][r] = (br < N && gk < K) ? b0[static_cast<size_t>(br) * K + gk] : 0.0f;
      if (SWIGLU) Bs1[kk][r] = (br < N && gk < K) ? b1[static_cast<size_t>(br) * K + gk] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float av[4], bv0[4], bv1[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        av[i] = As[kk][ty * 4 + i];
        bv0[i] = Bs0[kk][tx * 4 + i];
        if (SWIGLU) bv1[i] = Bs1[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc0[i][j] = fmaf(av[i], bv0[j], acc0[i][j]);
          if (SWIGLU) acc1[i][j] = fmaf(av[i], bv1[j], acc1[i][j]);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gr = row0 + ty * 4 + i;
    if (gr >= row_end) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gc = n0 + tx * 4 + j;
      if (gc >= N) continue;
      float v = acc0[i][j];
      if (SWIGLU) v = (v / (1.0f + expf(-v))) * acc1[i][j];
      out[static_cast<size_t>(gr) * N + gc] = v;
    }
  }
}

dim3 grid_for(int Tk, int E, int N) {
  // Upper bound on row blocks: every expert may end in a partial block.
  const int mblocks = (Tk + BM - 1) / BM + E;
  return dim3((N + BN - 1) / BN, mblocks);
}

}  // namespace

cudaError_t launch_ffn_f32_gate_up(const float* x_perm, const int32_t* offsets, const float* W1, const float* W3,
                                   float* h, int Tk, int d, int dff, int E, const Ctx& c, cudaStream_t s) {
  (void)c;
  launch_pdl(ffn_f32_kernel<true>, grid_for(Tk, E, dff), kThreads, 0, s, x_perm, offsets, W1, W3, h, Tk, E, d, dff, dff);
  return cudaGetLastError();
}

cudaError_t launch_ffn_f32_down(const float* h, const int32_t* offsets, const float* W2, float* y, int Tk, int d,
                                int dff, int E, const Ctx& c, cudaStream_t s) {
  (void)c;
  launch_pdl(ffn_f32_kernel<false>, grid_for(Tk, E, d), kThreads, 0, s, h, offsets, W2, nullptr, y, Tk, E, dff, d, d);
  return cudaGetLastError();
}

}  // namespace moe
