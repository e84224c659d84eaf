// Steps a0-a2 of the sparse-MoE layer: RMSNorm prologue (block form) and the
// router ("The Evolving Transformer - 05 Mixtral", section 03 RMSNorm and
// section 05 MoERouter).
//
// Router: a group of 32-256 threads per token (one warp for large batches,
// up to a whole CTA for small ones).  Each thread accumulates fp32 partial dot
// products of its 16-byte slices of x[t] with every gate row; a butterfly
// all-reduce inside each warp and a fixed-order sum over the group's warps
// give every thread all E logits, and every thread then runs the same top-k
// (descending, equal logits keep the lower index) and the softmax over the k
// chosen logits.  The summation order depends on the group size, so logits
// can differ in the last fp32 bit between batch sizes.  The page's order - softmax over all E, top-k, renormalise -
// gives the same weights because the normaliser over all E cancels.
#include <math.h>

#include "moe_internal.cuh"
#include "vec.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

// TPT threads cooperate on one token (a warp, or several warps of the CTA
// when the batch is too small to fill the GPU with one warp per token).
template <int EMAX, int TPT, typename TIn>
__global__ void __launch_bounds__(kThreads) router_topk_kernel(const TIn* __restrict__ x, const TIn* __restrict__ Wg,
                                                               int T, int d, int E, int k, int32_t* __restrict__ idx,
                                                               float* __restrict__ w, float* __restrict__ logits) {
  pdl_enter();
  constexpr int V = VecOf<TIn>::n;
  constexpr int WPT = TPT / 32;              // warps per token
  constexpr int TOK_PER_BLOCK = kThreads / TPT;
  __shared__ float part[WPT > 1 ? kThreads / 32 : 1][EMAX];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int slot = threadIdx.x / TPT;        // token of this thread within the block
  const int tt = threadIdx.x % TPT;          // thread within the token
  for (int base = blockIdx.x * TOK_PER_BLOCK; base < T; base += gridDim.x * TOK_PER_BLOCK) {
    const int t = base + slot;
    const bool valid = t < T;                // uniform across each warp (TPT >= 32)
    float acc[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) acc[e] = 0.0f;
    if (valid) {
      const TIn* xr = x + static_cast<size_t>(t) * d;
      for (int c = tt * V; c < d; c += TPT * V) {
        float xv[V];
        load_vec(xr + c, xv);
#pragma unroll
        for (int e = 0; e < EMAX; ++e) {
          if (e < E) {
            float gv[V];
            load_vec(Wg + static_cast<size_t>(e) * d + c, gv);
#pragma unroll
            for (int i = 0; i < V; ++i) acc[e] = fmaf(xv[i], gv[i], acc[e]);
          }
        }
      }
    }
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
      if (e < E) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[e] += __shfl_xor_sync(0xFFFFFFFFu, acc[e], o);
      }
    }
    if (WPT > 1) {
      if (lane == 0) {
#pragma unroll
        for (int e = 0; e < EMAX; ++e) part[warp][e] = acc[e];
      }
      __syncthreads();
      const int w0 = slot * WPT;
#pragma unroll
      for (int e = 0; e < EMAX; ++e) {
        float s = part[w0][e];
#pragma unroll
        for (int q = 1; q < WPT; ++q) s += part[w0 + q][e];
        acc[e] = s;
      }
      __syncthreads();
    }
    if (!valid) continue;
    // Top-k, identical in every thread of the token.  Strict '>' over
    // ascending e keeps the lower index on equal logits.  A NaN logit is
    // taken only when no other expert is left: any number replaces a NaN
    // best, and no comparison with a NaN candidate succeeds.
    uint64_t taken = 0;
    float sel_l[8];
    int sel_i[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      sel_l[j] = 0.0f;
      sel_i[j] = 0;
      if (j < k) {
        float best = 0.0f;
        int bi = -1;
#pragma unroll
        for (int e = 0; e < EMAX; ++e) {
          if (e < E && !((taken >> e) & 1ull) && (bi < 0 || acc[e] > best || (best != best && acc[e] == acc[e]))) {
            best = acc[e];
            bi = e;
          }
        }
        taken |= 1ull << bi;
        sel_l[j] = best;
        sel_i[j] = bi;
      }
    }
    // Softmax over the k chosen logits, shifted by the largest.
    float ex[8];
    float sum = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      ex[j] = (j < k) ? expf(sel_l[j] - sel_l[0]) : 0.0f;
      sum += ex[j];
    }
    if (tt < k) {
      float my_e = 0.0f;
      int my_i = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j == tt) {
          my_e = ex[j];
          my_i = sel_i[j];
        }
      }
      idx[static_cast<size_t>(t) * k + tt] = my_i;
      w[static_cast<size_t>(t) * k + tt] = my_e / sum;
    }
    if (logits != nullptr) {
      // Every thread of the token holds all E logits; thread tt writes
      // experts tt, tt + TPT, ... (E may exceed the group's 32 threads).
#pragma unroll
      for (int e = 0; e < EMAX; ++e) {
        if (e < E && e % TPT == tt) logits[static_cast<size_t>(t) * E + e] = acc[e];
      }
    }
  }
}

// RMSNorm, one warp per row: fp32 mean of squares, xn = x * r * gamma with
// r = 1 / sqrt(mean + eps), rounded once to the storage type.
template <typename TIn>
__global__ void __launch_bounds__(kThreads) rmsnorm_kernel(const TIn* __restrict__ x, const TIn* __restrict__ gamma,
                                                           float eps, TIn* __restrict__ xn, int T, int d) {
  pdl_enter();
  constexpr int V = VecOf<TIn>::n;
  const int lane = threadIdx.x & 31;
  const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int t = gwarp; t < T; t += nwarps) {
    const TIn* xr = x + static_cast<size_t>(t) * d;
    float ss = 0.0f;
    for (int c = lane * V; c < d; c += 32 * V) {
      float v[V];
      load_vec(xr + c, v);
#pragma unroll
      for (int i = 0; i < V; ++i) ss = fmaf(v[i], v[i], ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    const float r = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
    TIn* outr = xn + static_cast<size_t>(t) * d;
    for (int c = lane * V; c < d; c += 32 * V) {
      float v[V], g[V];
      load_vec(xr + c, v);
      load_vec(gamma + c, g);
#pragma unroll
      for (int i = 0; i < V; ++i) v[i] = (v[i] * r) * g[i];
      store_vec(outr + c, v);
    }
  }
}

int grid_for(int warps_needed, const Ctx& c) {
  const int per_block = kThreads / 32;
  int blocks = (warps_needed + per_block - 1) / per_block;
  const int cap = c.num_sms * 8;
  if (blocks > cap) blocks = cap;
  return blocks < 1 ? 1 : blocks;
}

// Threads per token: one warp when the batch fills the GPU with warps,
// up to a whole CTA for small batches (decode), so that every token's dot
// products are spread over enough threads to keep loads in flight.
int threads_per_token(int T, const Ctx& c) {
  int tpt = 32;
  while (tpt < kThreads && static_cast<long long>(T) * tpt < static_cast<long long>(c.num_sms) * 2048) tpt *= 2;
  return tpt;
}

template <int EMAX, typename TIn>
void launch_router_e(const TIn* xp, const TIn* gp, int T, int d, int E, int k, int32_t* idx, float* w, float* logits,
                     const Ctx& c, cudaStream_t s) {
  const int tpt = threads_per_token(T, c);
  const int per_block = kThreads / tpt;
  int grid = (T + per_block - 1) / per_block;
  const int cap = c.num_sms * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  switch (tpt) {
    case 32: launch_pdl(router_topk_kernel<EMAX, 32, TIn>, grid, kThreads, 0, s, xp, gp, T, d, E, k, idx, w, logits); break;
    case 64: launch_pdl(router_topk_kernel<EMAX, 64, TIn>, grid, kThreads, 0, s, xp, gp, T, d, E, k, idx, w, logits); break;
    case 128: launch_pdl(router_topk_kernel<EMAX, 128, TIn>, grid, kThreads, 0, s, xp, gp, T, d, E, k, idx, w, logits); break;
    default: launch_pdl(router_topk_kernel<EMAX, 256, TIn>, grid, kThreads, 0, s, xp, gp, T, d, E, k, idx, w, logits); break;
  }
}

template <typename TIn>
cudaError_t launch_router_t(const void* x, const void* Wg, int T, int d, int E, int k, int32_t* idx, float* w,
                            float* logits, const Ctx& c, cudaStream_t s) {
  const TIn* xp = static_cast<const TIn*>(x);
  const TIn* gp = static_cast<const TIn*>(Wg);
  if (E <= 8) {
    launch_router_e<8, TIn>(xp, gp, T, d, E, k, idx, w, logits, c, s);
  } else if (E <= 16) {
    launch_router_e<16, TIn>(xp, gp, T, d, E, k, idx, w, logits, c, s);
  } else if (E <= 32) {
    launch_router_e<32, TIn>(xp, gp, T, d, E, k, idx, w, logits, c, s);
  } else {
    launch_router_e<64, TIn>(xp, gp, T, d, E, k, idx, w, logits, c, s);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const void* x, const void* Wg, int T, int d, int E, int k, int32_t* idx, float* w,
                          float* logits, int dtype, const Ctx& c, cudaStream_t s) {
  if (dtype == MOE_DTYPE_BF16) return launch_router_t<__nv_bfloat16>(x, Wg, T, d, E, k, idx, w, logits, c, s);
  return launch_router_t<float>(x, Wg, T, d, E, k, idx, w, logits, c, s);
}

cudaError_t launch_rmsnorm(const void* x, const void* gamma, float eps, void* xn, int T, int d, int dtype,
                           const Ctx& c, cudaStream_t s) {
  const int grid = grid_for(T, c);
  if (dtype == MOE_DTYPE_BF16) {
    launch_pdl(rmsnorm_kernel<__nv_bfloat16>, grid, kThreads, 0, s, static_cast<const __nv_bfloat16*>(x),
                                                            static_cast<const __nv_bfloat16*>(gamma), eps,
                                                            static_cast<__nv_bfloat16*>(xn), T, d);
  } else {
    launch_pdl(rmsnorm_kernel<float>, grid, kThreads, 0, s, static_cast<const float*>(x), static_cast<const float*>(gamma),
                                                    eps, static_cast<float*>(xn), T, d);
  }
  return cudaGetLastError();
}

}  // namespace moe
