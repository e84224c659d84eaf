// Step a3 of the sparse-MoE layer: dispatch the (token, slot) pairs into
// expert-contiguous order ("The Evolving Transformer - 05 Mixtral", section 05:
// class MoE sends each expert the tokens routed to it; the page notes that
// production stacks batch the tokens of each expert together).
//
// rank kernel (one CTA): histogram of the expert indices, exclusive prefix
// sum into offsets[E+1], then a stable rank of every pair inside its expert.
// Pairs are taken in chunks of 1024 in ascending flat index f = t*k + j;
// inside a warp, __match_any_sync groups the lanes that picked the same
// expert and a popcount of the lower lanes gives the rank; per-warp counts
// in shared memory give the offset of each warp.  So the rows of an expert
// follow ascending f: ascending token, then slot.
//
// gather kernel (many CTAs): x_perm[p] = x[row_src[p]], a flat grid-stride
// loop over 16-byte chunks of the permuted rows.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kRankThreads = 1024;

template <int EMAX>
__global__ void __launch_bounds__(kRankThreads) dispatch_rank_kernel(const int32_t* __restrict__ idx, int Tk, int E,
                                                                     int k, int32_t* __restrict__ counts,
                                                                     int32_t* __restrict__ offsets,
                                                                     int32_t* __restrict__ row_src,
                                                                     int32_t* __restrict__ slot_pos, int* status) {
  pdl_enter();
  __shared__ int cnt[EMAX];
  __shared__ int cur[EMAX];
  __shared__ int wc[kRankThreads / 32][EMAX];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  for (int e = tid; e < EMAX; e += kRankThreads) cnt[e] = 0;
  for (int i = tid; i < (kRankThreads / 32) * EMAX; i += kRankThreads) (&wc[0][0])[i] = 0;
  __syncthreads();
  for (int f = tid; f < Tk; f += kRankThreads) {
    const int e = idx[f];
    if (e >= 0 && e < E) {
      atomicAdd(&cnt[e], 1);
    } else {
      record_status(status, MOE_EDEVICE);
    }
  }
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int e = 0; e < E; ++e) {
      offsets[e] = run;
      counts[e] = cnt[e];
      cur[e] = run;
      run += cnt[e];
    }
    offsets[E] = run;
  }
  __syncthreads();

  for (int base = 0; base < Tk; base += kRankThreads) {
    const int f = base + tid;
    int e = -1;
    if (f < Tk) {
      e = idx[f];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && lane == __ffs(peers) - 1) wc[warp][e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int pre = 0;
      for (int w2 = 0; w2 < warp; ++w2) pre += wc[w2][e];
      const int pos = cur[e] + pre + rank;
      slot_pos[f] = pos;
      row_src[pos] = f / k;
    } else if (f < Tk) {
      slot_pos[f] = -1;
    }
    __syncthreads();
    if (tid < E) {
      int s = 0;
      for (int w2 = 0; w2 < kRankThreads / 32; ++w2) s += wc[w2][tid];
      cur[tid] += s;
    }
    __syncthreads();
    for (int i = tid; i < (kRankThreads / 32) * EMAX; i += kRankThreads) (&wc[0][0])[i] = 0;
    __syncthreads();
  }
}

constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(const uint4* __restrict__ x,
                                                                     const int32_t* __restrict__ row_src,
                                                                     uint4* __restrict__ x_perm, int Tk, int T,
                                                                     int vecs_per_row, int* status) {
  pdl_enter();
  const long long total = static_cast<long long>(Tk) * vecs_per_row;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int p = static_cast<int>(i / vecs_per_row);
    const int v = static_cast<int>(i - static_cast<long long>(p) * vecs_per_row);
    const int t = __ldg(row_src + p);
    if (t < 0 || t >= T) {
      if (v == 0) record_status(status, MOE_EDEVICE);
      continue;
    }
    x_perm[i] = __ldg(x + static_cast<size_t>(t) * vecs_per_row + v);
  }
}

}  // namespace

cudaError_t launch_dispatch(const int32_t* idx, int Tk, int E, int k, int32_t* counts, int32_t* offsets,
                            int32_t* row_src, int32_t* slot_pos, const Ctx& c, cudaStream_t s) {
  if (E <= 8) {
    launch_pdl(dispatch_rank_kernel<8>, 1, kRankThreads, 0, s, idx, Tk, E, k, counts, offsets, row_src, slot_pos, c.status);
  } else {
    launch_pdl(dispatch_rank_kernel<64>, 1, kRankThreads, 0, s, idx, Tk, E, k, counts, offsets, row_src, slot_pos, c.status);
  }
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* x, const int32_t* row_src, void* x_perm, int T, int Tk,
                               size_t row_bytes, const Ctx& c, cudaStream_t s) {
  const int vecs = static_cast<int>(row_bytes / 16);
  long long blocks = (static_cast<long long>(Tk) * vecs + kGatherThreads - 1) / kGatherThreads;
  const int cap = c.num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  launch_pdl(gather_rows_kernel, static_cast<int>(blocks), kGatherThreads, 0, s, static_cast<const uint4*>(x), row_src,
                                                       static_cast<uint4*>(x_perm), Tk, T, vecs, c.status);
  return cudaGetLastError();
}

}  // namespace moe
