// Step a6 of the sparse-MoE layer: gate-weighted combine of each token's k
// expert outputs, fused with the un-permute and (block form) the residual add
// ("The Evolving Transformer - 05 Mixtral", section 05, class MoE: each chosen
// expert's output is added with its weight; section 06, Block: x + MoE(...);
// Mixtral 8x7B model reference page, Architecture: the chosen experts'
// outputs are combined additively).
//
// Every thread owns one 16-byte chunk of one token's output row (a flat
// grid-stride loop over T x d/8 chunks, so small batches still spread over
// the GPU): out[t] = sum_j w[t,j] * y_perm[slot_pos[t*k+j]] in fp32, slot
// order, then + residual[t], rounded once to the storage type.
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
  pdl_enter();
  constexpr int V = VecOf<TIo>::n;
  const int vecs = d / V;
  const long long total = static_cast<long long>(T) * vecs;
  const long long Tk = static_cast<long long>(T) * k;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / vecs);
    const int c = static_cast<int>(i - static_cast<long long>(t) * vecs) * V;
    float acc[V];
#pragma unroll
    for (int q = 0; q < V; ++q) acc[q] = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < k) {
        const int p = __ldg(slot_pos + static_cast<size_t>(t) * k + j);
        if (p >= 0 && p < Tk) {
          const float wt = __ldg(w + static_cast<size_t>(t) * k + j);
          float v[V];
          load_vec(y + static_cast<size_t>(p) * d + c, v);
#pragma unroll
          for (int q = 0; q < V; ++q) acc[q] = fmaf(wt, v[q], acc[q]);
        } else if (c == 0) {
          record_status(status, MOE_EDEVICE);
        }
      }
    }
    if (residual != nullptr) {
      float r[V];
      load_vec(residual + static_cast<size_t>(t) * d + c, r);
#pragma unroll
      for (int q = 0; q < V; ++q) acc[q] += r[q];
    }
    store_vec(out + static_cast<size_t>(t) * d + c, acc);
  }
}

}  // namespace

cudaError_t launch_combine(const void* y, const int32_t* slot_pos, const float* w, const void* residual, void* out,
                           int T, int d, int k, int dtype, const Ctx& c, cudaStream_t s) {
  const long long items = static_cast<long long>(T) * (d / (dtype == MOE_DTYPE_BF16 ? 8 : 4));
  long long blocks = (items + kThreads - 1) / kThreads;
  const int cap = c.num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (dtype == MOE_DTYPE_BF16) {
    launch_pdl(combine_kernel<__nv_bfloat16>, static_cast<int>(blocks), kThreads, 0, s, 
        static_cast<const __nv_bfloat16*>(y), slot_pos, w, static_cast<const __nv_bfloat16*>(residual),
        static_cast<__nv_bfloat16*>(out), T, d, k, c.status);
  } else {
    launch_pdl(combine_kernel<float>, static_cast<int>(blocks), kThreads, 0, s, static_cast<const float*>(y), slot_pos, w,
                                                      static_cast<const float*>(residual), static_cast<float*>(out),
                                                      T, d, k, c.status);
  }
  return cudaGetLastError();
}

}  // namespace moe
