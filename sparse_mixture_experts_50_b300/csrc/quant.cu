// Weight-only int8 quantisation of the expert matrices (KerasFormers Mixtral
// docs, "Lower memory": checkpoints load with the weights alone quantised to
// int8 while activations stay bf16).  The docs leave the scheme open; this
// library uses symmetric per-output-channel codes: each row of an nn.Linear
// weight W[rows, cols] gets one fp32 scale s = max|row| / 127 and int8 codes
// q = round-half-even(w / s) clamped to [-127, 127]; a row of zeros gets s = 0
// and q = 0.  The matrix the layer then multiplies by is s[row] * q[row, col].
//
// Both the scale and every code come from IEEE fp32 divisions rounded to
// nearest, so the codes are reproducible bit for bit by any IEEE fp32
// implementation of the same two steps.
//
// One warp per row, a grid-stride loop over rows: pass 1 reduces max|w| over
// the row with 16-byte loads, pass 2 re-reads the row (from L1/L2) and writes
// 8 codes per 8-byte store.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void bf16x8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__global__ void __launch_bounds__(kThreads) quantize_rows_int8_kernel(const __nv_bfloat16* __restrict__ W,
                                                                     long long rows, int cols,
                                                                     int8_t* __restrict__ q,
                                                                     float* __restrict__ scale) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (kThreads / 32);
  for (long long row = static_cast<long long>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    const __nv_bfloat16* src = W + row * cols;
    float amax = 0.0f;
    for (int c = lane * 8; c < cols; c += 32 * 8) {
      float v[8];
      bf16x8(src + c, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float s = __fdiv_rn(amax, 127.0f);
    int8_t* dst = q + row * cols;
    for (int c = lane * 8; c < cols; c += 32 * 8) {
      float v[8];
      bf16x8(src + c, v);
      uint32_t pk[2] = {0u, 0u};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        int qi = 0;
        if (s > 0.0f) {
          qi = __float2int_rn(__fdiv_rn(v[i], s));
          qi = qi > 127 ? 127 : (qi < -127 ? -127 : qi);
        }
        pk[i >> 2] |= (static_cast<uint32_t>(qi) & 0xFFu) << (8 * (i & 3));
      }
      *reinterpret_cast<uint2*>(dst + c) = make_uint2(pk[0], pk[1]);
    }
    if (lane == 0) scale[row] = s;
  }
}

}  // namespace

cudaError_t launch_quantize_int8(const void* W, long long rows, int cols, int8_t* q, float* scale, const Ctx& c,
                                 cudaStream_t s) {
  long long blocks = (rows + kThreads / 32 - 1) / (kThreads / 32);
  const long long cap = static_cast<long long>(c.num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  launch_pdl(quantize_rows_int8_kernel, static_cast<int>(blocks), kThreads, 0, s,
             static_cast<const __nv_bfloat16*>(W), rows, cols, q, scale);
  return cudaGetLastError();
}

}  // namespace moe
