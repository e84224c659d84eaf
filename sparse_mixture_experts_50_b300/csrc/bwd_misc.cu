// Backward of the router, dispatch and combine steps of the sparse-MoE layer
// (Mixtral 8x7B model reference page, Training: experts and router are
// trained together; "The Evolving Transformer - 05 Mixtral", section 05:
// out[t] = sum_j w[t,j] y_j[t], (w, i) = softmax over the k largest logits of
// x Wg^T), and the layout changes the expert-GEMM backward needs.
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
//   transposes: batched [B, R, C] -> [B, C, R] for the weights, and
//            token-major [Tk, C] -> [C, Kp] with each expert's tokens padded
//            to a multiple of 64 (zeros), for the weight-gradient GEMMs.
#include "moe_internal.cuh"
#include "vec.cuh"

namespace moe {
namespace {

constexpr int kKpad = 64;
constexpr int kMaxE = 64;

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
// Block (column block of 256, token chunk): per-expert sums of dl * x for its
// columns over its tokens, in shared memory (each thread owns a column).
__global__ void __launch_bounds__(256) dwg_partial_kernel(const __nv_bfloat16* __restrict__ x,
                                                          const int32_t* __restrict__ idx,
                                                          const float* __restrict__ dl, float* __restrict__ part,
                                                          int T, int d, int E, int k, int chunk) {
  extern __shared__ float accs[];  // [E][256]
  pdl_enter();
  const int c = blockIdx.x * 256 + threadIdx.x;
  const int t0 = blockIdx.y * chunk;
  const int t1 = min(T, t0 + chunk);
  for (int e = 0; e < E; ++e) accs[e * 256 + threadIdx.x] = 0.0f;
  if (c < d) {
    for (int t = t0; t < t1; ++t) {
      const float xv = __bfloat162float(x[static_cast<size_t>(t) * d + c]);
      for (int j = 0; j < k; ++j) {
        const size_t f = static_cast<size_t>(t) * k + j;
        const int e = idx[f];
        if (e >= 0 && e < E) accs[e * 256 + threadIdx.x] = fmaf(dl[f], xv, accs[e * 256 + threadIdx.x]);
      }
    }
    for (int e = 0; e < E; ++e)
      part[(static_cast<size_t>(blockIdx.y) * E + e) * d + c] = accs[e * 256 + threadIdx.x];
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

// ---------------------------------------------------------------- transposes
// 64 x 64 tiles through shared memory with 16-byte global accesses: each
// thread loads 8 consecutive columns of a source row, and writes 8
// consecutive rows of one column as a 16-byte run of a destination row
// (a warp's lanes take 32 consecutive columns, so its shared-memory reads of
// one row are conflict-free).
constexpr int kTp = 72;  // tile row pitch in elements (144 bytes, 16-byte aligned)

__device__ __forceinline__ void tile_store_out(const __nv_bfloat16 (*tile)[kTp], __nv_bfloat16* dst_row, int col,
                                               int r0, int rows_ok) {
  // dst_row points at destination row `col`; writes rows r0 .. r0+7 of the tile's column.
  uint32_t w[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint16_t lo = __bfloat16_as_ushort(tile[r0 + 2 * m][col]);
    const uint16_t hi = __bfloat16_as_ushort(tile[r0 + 2 * m + 1][col]);
    w[m] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  if (rows_ok >= 8) {
    *reinterpret_cast<uint4*>(dst_row) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    for (int m = 0; m < rows_ok; ++m)
      dst_row[m] = __ushort_as_bfloat16(static_cast<uint16_t>(w[m >> 1] >> (16 * (m & 1))));
  }
}

// [B, R, C] -> [B, C, R].  C % 8 == 0 and R % 8 == 0.
__global__ void __launch_bounds__(256) transpose_batched_kernel(const __nv_bfloat16* __restrict__ src,
                                                                __nv_bfloat16* __restrict__ dst, int R, int C) {
  __shared__ __align__(16) __nv_bfloat16 tile[64][kTp];
  pdl_enter();
  const size_t b = blockIdx.z;
  const int r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
  const __nv_bfloat16* s = src + b * R * C;
  __nv_bfloat16* o = dst + b * R * C;
  for (int i = threadIdx.x; i < 64 * 8; i += 256) {
    const int r = i >> 3, q = (i & 7) * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r0 + r < R && c0 + q < C) v = __ldg(reinterpret_cast<const uint4*>(s + static_cast<size_t>(r0 + r) * C + c0 + q));
    *reinterpret_cast<uint4*>(&tile[r][q]) = v;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, wv = threadIdx.x >> 5;  // 8 warps
  for (int i = wv; i < 2 * 8; i += 8) {
    const int col = (i & 1) * 32 + lane;   // tile column = destination row
    const int rq = (i >> 1) * 8;           // 8 tile rows = 8 destination columns
    if (c0 + col < C && r0 + rq < R)
      tile_store_out(tile, o + static_cast<size_t>(c0 + col) * R + r0 + rq, col, rq, R - (r0 + rq));
  }
}

// Token-major [Tk, C] (rows grouped by expert) -> [C, Kp]: token p of expert
// e goes to column kseg[e] + p - offsets[e]; every other column is zero.
// C % 8 == 0, Kp % 64 == 0.
__global__ void __launch_bounds__(256) transpose_segments_kernel(const __nv_bfloat16* __restrict__ src,
                                                                 const int32_t* __restrict__ offsets,
                                                                 __nv_bfloat16* __restrict__ dst, int Tk, int C,
                                                                 int Kp, int E) {
  __shared__ __align__(16) __nv_bfloat16 tile[64][kTp];
  __shared__ int off_s[kMaxE + 1];
  __shared__ int kseg_s[kMaxE + 1];
  __shared__ int srow[64];
  pdl_enter();
  if (threadIdx.x == 0) {
    int prev = 0, ks = 0;
    for (int e = 0; e <= E; ++e) {
      int o = offsets[e];
      if (o < prev || o > Tk) o = prev;  // a bad table was reported by the forward; treated as empty
      if (e > 0) ks += (o - prev + kKpad - 1) / kKpad * kKpad;
      off_s[e] = o;
      kseg_s[e] = ks;
      prev = o;
    }
  }
  __syncthreads();
  const int k0 = blockIdx.x * 64, c0 = blockIdx.y * 64;
  if (threadIdx.x < 64) {
    const int kk = k0 + threadIdx.x;
    int p = -1;
    if (kk < kseg_s[E]) {
      int e = 0;
      while (e + 1 < E && kseg_s[e + 1] <= kk) ++e;
      const int local = kk - kseg_s[e];
      if (local < off_s[e + 1] - off_s[e]) p = off_s[e] + local;
    }
    srow[threadIdx.x] = p;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 64 * 8; i += 256) {
    const int r = i >> 3, q = (i & 7) * 8;
    const int p = srow[r];
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (p >= 0 && c0 + q < C) v = __ldg(reinterpret_cast<const uint4*>(src + static_cast<size_t>(p) * C + c0 + q));
    *reinterpret_cast<uint4*>(&tile[r][q]) = v;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, wv = threadIdx.x >> 5;
  for (int i = wv; i < 2 * 8; i += 8) {
    const int col = (i & 1) * 32 + lane;   // channel = destination row
    const int rq = (i >> 1) * 8;           // 8 padded-token columns
    if (c0 + col < C && k0 + rq < Kp)
      tile_store_out(tile, dst + static_cast<size_t>(c0 + col) * Kp + k0 + rq, col, rq, Kp - (k0 + rq));
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

int dwg_chunks(int T) { return T < 64 ? 1 : (T + 255) / 256 < 64 ? (T + 255) / 256 : 64; }

cudaError_t launch_dwg(const void* x, const int32_t* idx, const float* dl, float* part, float* dWg, int T, int d, int E,
                       int k, const Ctx& c, cudaStream_t s) {
  const int nch = dwg_chunks(T);
  const int chunk = (T + nch - 1) / nch;
  dim3 grid((d + 255) / 256, nch);
  const size_t smem = static_cast<size_t>(E) * 256 * sizeof(float);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(dwg_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
          cudaSuccess)
    return cudaGetLastError();
  launch_pdl(dwg_partial_kernel, grid, dim3(256), smem, s, static_cast<const __nv_bfloat16*>(x), idx, dl, part, T, d,
             E, k, chunk);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int Ed = E * d;
  int blocks = (Ed + 255) / 256;
  if (blocks > c.num_sms * 8) blocks = c.num_sms * 8;
  launch_pdl(dwg_reduce_kernel, blocks, 256, 0, s, static_cast<const float*>(part), dWg, nch, Ed);
  return cudaGetLastError();
}

cudaError_t launch_transpose_batched(const void* src, void* dst, int B, int R, int C, cudaStream_t s) {
  dim3 grid((C + 63) / 64, (R + 63) / 64, B);
  launch_pdl(transpose_batched_kernel, grid, dim3(256), 0, s, static_cast<const __nv_bfloat16*>(src),
             static_cast<__nv_bfloat16*>(dst), R, C);
  return cudaGetLastError();
}

cudaError_t launch_transpose_segments(const void* src, const int32_t* offsets, void* dst, int Tk, int C, int Kp,
                                      int E, cudaStream_t s) {
  dim3 grid((Kp + 63) / 64, (C + 63) / 64);
  launch_pdl(transpose_segments_kernel, grid, dim3(256), 0, s, static_cast<const __nv_bfloat16*>(src), offsets,
             static_cast<__nv_bfloat16*>(dst), Tk, C, Kp, E);
  return cudaGetLastError();
}

}  // namespace moe
