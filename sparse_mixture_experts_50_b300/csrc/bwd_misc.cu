// Backward of the router, dispatch and combine steps of the sparse-MoE layer
// (Mixtral 8x7B model reference page, Training: experts and router are
// trained together; "The Evolving Transformer - 05 Mixtral", section 05:
// out[t] = sum_j w[t,j] y_j[t], (w, i) = softmax over the k largest logits of
// x Wg^T).
//
//   route:   for p = slot_pos[t*k+j]: dout_perm[p] = dout[t] (an exact copy),
//            w_perm[p] = w[t,j], dy_perm[p] = w[t,j] dout[t] (rounded, for
//            the W2 gradient) and dw[t,j] = <dout[t], y_perm[p]>; then the
//            softmax over the k chosen logits gives
//            dl[t,j] = w[t,j] (dw[t,j] - sum_i w[t,i] dw[t,i]).
//   dx:      dx[t] = sum_j dx_perm[slot_pos[t*k+j]] + sum_j dl[t,j] Wg[i[t,j]]
//   dWg:     dWg[e] = sum over (t, j) with i[t,j] = e of dl[t,j] x[t], in
//            two deterministic stages (per-chunk partial sums, then their
//            sum in chunk order).
#include "moe_internal.cuh"
#include "vec.cuh"

namespace moe {
namespace {


// ---------------------------------------------------------------- route
// One warp per token.
__global__ void __launch_bounds__(256) route_bwd_kernel(const __nv_bfloat16* __restrict__ dout,
                                                        const __nv_bfloat16* __restrict__ y_perm,
                                                        const int32_t* __restrict__ slot_pos,
                                                        const float* __restrict__ w, __nv_bfloat16* __restrict__ dy_perm,
                                                        __nv_bfloat16* __restrict__ dout_perm,
                                                        float* __restrict__ w_perm, float* __restrict__ dl, int T, int d,
                                                        int k, int* status) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const long long Tk = static_cast<long long>(T) * k;
  float dw[8];
  float wt[8];
  const __nv_bfloat16* g = dout + static_cast<size_t>(t) * d;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    dw[j] = 0.0f;
    wt[j] = 0.0f;
    if (j >= k) continue;
    const int p = slot_pos[static_cast<size_t>(t) * k + j];
    wt[j] = w[static_cast<size_t>(t) * k + j];
    if (p < 0 || p >= Tk) {
      if (lane == 0) record_status(status, MOE_EDEVICE);
      continue;
    }
    const __nv_bfloat16* y = y_perm + static_cast<size_t>(p) * d;
    __nv_bfloat16* dy = dy_perm + static_cast<size_t>(p) * d;
    __nv_bfloat16* dp = dout_perm + static_cast<size_t>(p) * d;
    if (lane == 0) w_perm[p] = wt[j];
    float s = 0.0f;
    for (int c = lane * 8; c < d; c += 256) {
      float gv[8], yv[8], o[8];
      load_vec(g + c, gv);
      load_vec(y + c, yv);
      *reinterpret_cast<uint4*>(dp + c) = *reinterpret_cast<const uint4*>(g + c);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        s = fmaf(gv[q], yv[q], s);
        o[q] = wt[j] * gv[q];
      }
      store_vec(dy + c, o);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
    dw[j] = s;
  }
  float mean = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) mean += wt[j] * dw[j];
  if (lane < k) {
    float v = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j == lane) v = wt[j] * (dw[j] - mean);
    dl[static_cast<size_t>(t) * k + lane] = v;
  }
}

// ---------------------------------------------------------------- dx
__global__ void __launch_bounds__(256) dx_gather_kernel(const __nv_bfloat16* __restrict__ dx_perm,
                                                        const int32_t* __restrict__ slot_pos,
                                                        const int32_t* __restrict__ idx, const float* __restrict__ dl,
                                                        const __nv_bfloat16* __restrict__ Wg, __nv_bfloat16* __restrict__ dx,
                                                        int T, int d, int E, int k, int* status) {
  pdl_enter();
  const int vecs = d / 8;
  const long long total = static_cast<long long>(T) * vecs;
  const long long Tk = static_cast<long long>(T) * k;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / vecs);
    const int c = static_cast<int>(i - static_cast<long long>(t) * vecs) * 8;
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
    for (int j = 0; j < k; ++j) {
      const size_t f = static_cast<size_t>(t) * k + j;
      const int p = slot_pos[f];
      const int e = idx[f];
      if (p < 0 || p >= Tk || e < 0 || e >= E) {
        if (c == 0) record_status(status, MOE_EDEVICE);
        continue;
      }
      float v[8], wg[8];
      load_vec(dx_perm + static_cast<size_t>(p) * d + c, v);
      load_vec(Wg + static_cast<size_t>(e) * d + c, wg);
      const float s = dl[f];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] += v[q] + s * wg[q];
    }
    store_vec(dx + static_cast<size_t>(t) * d + c, acc);
  }
}

// ---------------------------------------------------------------- dWg
// dWg = G^T x with G[t, e] = sum_j [i[t,j] = e] dl[t,j]: a [T, E] matrix with
// k nonzeros per row, so a small dense contraction over the tokens.  A block
// takes a chunk of tokens and 2048 columns; each thread owns 8 consecutive
// columns (one 16-byte load of x per token) and keeps 8 experts x 8 columns
// of fp32 sums in registers (experts in groups of 8).  The chunk's G rows
// are built in shared memory, kDwgSub tokens at a time, one thread per token
// adding its k entries in slot order.  Every sum runs in token order, and
// the chunks' partial sums are added in chunk order: the result does not
// depend on the launch shape's timing.
constexpr int kDwgThreads = 256;
constexpr int kDwgCols = 8;
constexpr int kDwgGroup = 8;
constexpr int kDwgSub = 64;

__global__ void __launch_bounds__(kDwgThreads) dwg_partial_kernel(const __nv_bfloat16* __restrict__ x,
                                                                  const int32_t* __restrict__ idx,
                                                                  const float* __restrict__ dl,
                                                                  float* __restrict__ part, int T, int d, int E, int k,
                                                                  int chunk) {
  extern __shared__ float G[];  // [kDwgSub][E]
  pdl_enter();
  const int t0 = blockIdx.y * chunk;
  const int t1 = min(T, t0 + chunk);
  const int c0 = (blockIdx.x * kDwgThreads + threadIdx.x) * kDwgCols;
  const bool live = c0 < d;
  for (int eg = 0; eg < E; eg += kDwgGroup) {
    float acc[kDwgGroup][kDwgCols];
#pragma unroll
    for (int e = 0; e < kDwgGroup; ++e)
#pragma unroll
      for (int q = 0; q < kDwgCols; ++q) acc[e][q] = 0.0f;
    for (int s0 = t0; s0 < t1; s0 += kDwgSub) {
      const int ns = min(kDwgSub, t1 - s0);
      __syncthreads();  // the previous sub-chunk's G is no longer read
      for (int i = threadIdx.x; i < kDwgSub * E; i += kDwgThreads) G[i] = 0.0f;
      __syncthreads();
      for (int t = threadIdx.x; t < ns; t += kDwgThreads) {
        for (int j = 0; j < k; ++j) {
          const size_t f = static_cast<size_t>(s0 + t) * k + j;
          const int e = __ldg(idx + f);
          if (e >= 0 && e < E) G[t * E + e] += __ldg(dl + f);
        }
      }
      __syncthreads();
      if (live) {
#pragma unroll 4
        for (int t = 0; t < ns; ++t) {
          float xv[kDwgCols];
          load_vec(x + static_cast<size_t>(s0 + t) * d + c0, xv);
#pragma unroll
          for (int e = 0; e < kDwgGroup; ++e) {
            const float g = eg + e < E ? G[t * E + eg + e] : 0.0f;
#pragma unroll
            for (int q = 0; q < kDwgCols; ++q) acc[e][q] = fmaf(g, xv[q], acc[e][q]);
          }
        }
      }
    }
    if (live) {
#pragma unroll
      for (int e = 0; e < kDwgGroup; ++e) {
        if (eg + e >= E) break;
        float* dst = part + (static_cast<size_t>(blockIdx.y) * E + eg + e) * d + c0;
        const float lo[4] = {acc[e][0], acc[e][1], acc[e][2], acc[e][3]};
        const float hi[4] = {acc[e][4], acc[e][5], acc[e][6], acc[e][7]};
        store_vec(dst, lo);
        store_vec(dst + 4, hi);
      }
    }
  }
}

__global__ void __launch_bounds__(256) dwg_reduce_kernel(const float* __restrict__ part, float* __restrict__ dWg,
                                                         int nchunks, int Ed) {
  pdl_enter();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < Ed; i += gridDim.x * blockDim.x) {
    float s = 0.0f;
    for (int ch = 0; ch < nchunks; ++ch) s += part[static_cast<size_t>(ch) * Ed + i];
    dWg[i] = s;
  }
}

}  // namespace

cudaError_t launch_route_bwd(const void* dout, const void* y_perm, const int32_t* slot_pos, const float* w,
                             void* dy_perm, void* dout_perm, float* w_perm, float* dl, int T, int d, int k,
                             const Ctx& c, cudaStream_t s) {
  launch_pdl(route_bwd_kernel, (T + 7) / 8, 256, 0, s, static_cast<const __nv_bfloat16*>(dout),
             static_cast<const __nv_bfloat16*>(y_perm), slot_pos, w, static_cast<__nv_bfloat16*>(dy_perm),
             static_cast<__nv_bfloat16*>(dout_perm), w_perm, dl, T, d, k, c.status);
  return cudaGetLastError();
}

cudaError_t launch_dx_gather(const void* dx_perm, const int32_t* slot_pos, const int32_t* idx, const float* dl,
                             const void* Wg, void* dx, int T, int d, int E, int k, const Ctx& c, cudaStream_t s) {
  const long long items = static_cast<long long>(T) * (d / 8);
  long long blocks = (items + 255) / 256;
  if (blocks > c.num_sms * 8LL) blocks = c.num_sms * 8LL;
  if (blocks < 1) blocks = 1;
  launch_pdl(dx_gather_kernel, static_cast<int>(blocks), 256, 0, s, static_cast<const __nv_bfloat16*>(dx_perm),
             slot_pos, idx, dl, static_cast<const __nv_bfloat16*>(Wg), static_cast<__nv_bfloat16*>(dx), T, d, E, k,
             c.status);
  return cudaGetLastError();
}

// Token chunks of dWg's first stage: ~64 tokens each, at most 64 chunks.
int dwg_chunks(int T) { return T <= 64 ? 1 : (T + 63) / 64 < 64 ? (T + 63) / 64 : 64; }

cudaError_t launch_dwg(const void* x, const int32_t* idx, const float* dl, float* part, float* dWg, int T, int d, int E,
                       int k, const Ctx& c, cudaStream_t s) {
  const int nch = dwg_chunks(T);
  const int chunk = (T + nch - 1) / nch;
  const int cols_per_block = kDwgThreads * kDwgCols;
  dim3 grid((d + cols_per_block - 1) / cols_per_block, nch);
  const size_t smem = static_cast<size_t>(kDwgSub) * E * sizeof(float);  // <= 16 KB (E <= 64)
  launch_pdl(dwg_partial_kernel, grid, dim3(kDwgThreads), smem, s, static_cast<const __nv_bfloat16*>(x), idx, dl, part,
             T, d, E, k, chunk);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int Ed = E * d;
  int blocks = (Ed + 255) / 256;
  if (blocks > c.num_sms * 8) blocks = c.num_sms * 8;
  launch_pdl(dwg_reduce_kernel, blocks, 256, 0, s, static_cast<const float*>(part), dWg, nch, Ed);
  return cudaGetLastError();
}

}  // namespace moe
