// Step a6 of the sparse-MoE layer: gate-weighted combine of each token's k
// expert outputs, fused with the un-permute and (block form) the residual add
// ("The Evolving Transformer - 05 Mixtral", section 05, class MoE: each chosen
// expert's output is added with its weight; section 06, Block: x + MoE(...);
// Mixtral 8x7B model reference page, Architecture: the chosen experts'
// outputs are combined additively).
//
// One warp per token: out[t] = sum_j w[t,j] * y_perm[slot_pos[t*k+j]] in fp32,
// slot order, then + residual[t], rounded once to the storage type.
#include "moe_internal.cuh"
#include "vec.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

template <typename TIo>
__global__ void __launch_bounds__(kThreads) combine_kernel(const TIo* __restrict__ y, const int32_t* __restrict__ slot_pos,
                                                           const float* __restrict__ w,
                                                           const TIo* __restrict__ residual, TIo* __restrict__ out,
                                                           int T, int d, int k, int* status) {
  constexpr int V = VecOf<TIo>::n;
  const int lane = threadIdx.x & 31;
  const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const long long Tk = static_cast<long long>(T) * k;
  for (int t = gwarp; t < T; t += nwarps) {
    int pos[8];
    float wt[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      pos[j] = -1;
      wt[j] = 0.0f;
      if (j < k) {
        const int p = slot_pos[static_cast<size_t>(t) * k + j];
        if (p >= 0 && p < Tk) {
          pos[j] = p;
          wt[j] = w[static_cast<size_t>(t) * k + j];
        } else if (lane == 0) {
          record_status(status, MOE_EDEVICE);
        }
      }
    }
    for (int c = lane * V; c < d; c += 32 * V) {
      float acc[V];
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (pos[j] >= 0) {
          float v[V];
          load_vec(y + static_cast<size_t>(pos[j]) * d + c, v);
#pragma unroll
          for (int i = 0; i < V; ++i) acc[i] = fmaf(wt[j], v[i], acc[i]);
        }
      }
      if (residual != nullptr) {
        float r[V];
        load_vec(residual + static_cast<size_t>(t) * d + c, r);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] += r[i];
      }
      store_vec(out + static_cast<size_t>(t) * d + c, acc);
    }
  }
}

}  // namespace

cudaError_t launch_combine(const void* y, const int32_t* slot_pos, const float* w, const void* residual, void* out,
                           int T, int d, int k, int dtype, const Ctx& c, cudaStream_t s) {
  const int per_block = kThreads / 32;
  int blocks = (T + per_block - 1) / per_block;
  const int cap = c.num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (dtype == MOE_DTYPE_BF16) {
    combine_kernel<__nv_bfloat16><<<blocks, kThreads, 0, s>>>(
        static_cast<const __nv_bfloat16*>(y), slot_pos, w, static_cast<const __nv_bfloat16*>(residual),
        static_cast<__nv_bfloat16*>(out), T, d, k, c.status);
  } else {
    combine_kernel<float><<<blocks, kThreads, 0, s>>>(static_cast<const float*>(y), slot_pos, w,
                                                      static_cast<const float*>(residual), static_cast<float*>(out),
                                                      T, d, k, c.status);
  }
  return cudaGetLastError();
}

}  // namespace moe
