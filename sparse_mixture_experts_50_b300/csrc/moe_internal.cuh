// Internal declarations shared by the libmoe translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "moe.h"

namespace moe {

// Per-call context: the device that owns the output, its SM count, the
// address of that device's status word and the spin-wait limit.
struct Ctx {
  int device;
  int num_sms;
  int* status;                 // device address of the per-device status word
  unsigned long long wait_ns;  // bounded-wait limit for spinning kernels
  int max_rows_per_expert;     // expert GEMMs: known bound on any expert's rows (0: only Tk)
};

// Sets the calling thread's current device to the one owning `dev_ptr`
// (or keeps the current device if the pointer is not a device pointer) and
// fills `ctx`; `*prev_device` receives the device that was current before
// (-1 if it could not be read).  Returns MOE_OK or MOE_ECUDA.
int make_ctx(const void* dev_ptr, Ctx* ctx, int* prev_device);

// What every entry point holds for its call: the context of the device that
// owns its operands, made current for the call, and the caller's current
// device, made current again when the entry point returns.
class CtxScope {
 public:
  CtxScope() = default;
  CtxScope(const CtxScope&) = delete;
  CtxScope& operator=(const CtxScope&) = delete;
  ~CtxScope() {
    if (prev_ >= 0 && switched_) cudaSetDevice(prev_);
  }
  int init(const void* dev_ptr) {
    const int rc = make_ctx(dev_ptr, &ctx_, &prev_);
    switched_ = prev_ >= 0;
    return rc;
  }
  const Ctx& ctx() const { return ctx_; }

 private:
  Ctx ctx_ = {};
  int prev_ = -1;
  bool switched_ = false;
};

// Records `code` in the device status word unless one is already recorded.
__device__ __forceinline__ void record_status(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// Programmatic dependent launch.  Every kernel of the layer lets the next
// launch on the stream start as soon as all its CTAs are running
// (launch_dependents), and waits for the previous one to finish, with its
// writes visible, before it touches global memory (wait).  The overlap hides
// launch latency and the tensor-core kernels' set-up.  With no programmatic
// predecessor the wait returns at once.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
  pdl_trigger();
  pdl_wait();
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- launchers (each returns a cudaError_t from the launch) --------------
cudaError_t launch_router(const void* x, const void* Wg, int T, int d, int E, int k,
                          int32_t* idx, float* w, float* logits, int dtype,
                          const Ctx& c, cudaStream_t s);
cudaError_t launch_rmsnorm(const void* x, const void* gamma, float eps, void* xn, int T, int d,
                           int dtype, const Ctx& c, cudaStream_t s);
cudaError_t launch_dispatch(const int32_t* idx, int Tk, int E, int k, int32_t* counts,
                            int32_t* offsets, int32_t* row_src, int32_t* slot_pos,
                            const Ctx& c, cudaStream_t s);
cudaError_t launch_gather_rows(const void* x, const int32_t* row_src, void* x_perm, int T, int Tk,
                               size_t row_bytes, const Ctx& c, cudaStream_t s);
cudaError_t launch_combine(const void* y, const int32_t* slot_pos, const float* w,
                           const void* residual, void* out, int T, int d, int k, int dtype,
                           const Ctx& c, cudaStream_t s);
cudaError_t launch_ffn_f32_gate_up(const float* x_perm, const int32_t* offsets, const float* W1,
                                   const float* W3, float* h, int Tk, int d, int dff, int E,
                                   const Ctx& c, cudaStream_t s);
cudaError_t launch_ffn_f32_down(const float* h, const int32_t* offsets, const float* W2, float* y,
                                int Tk, int d, int dff, int E, const Ctx& c, cudaStream_t s);
// bf16 tcgen05 path; returns MOE_* status (tensor-map encoding can fail).
// keep (optional): bf16 planes [2, Tk, dff] of p = b silu'(a) and
// q = silu(a), for the backward.
int launch_tc_gate_up(const void* x_perm, const int32_t* offsets, const void* W1, const void* W3,
                      void* h, int Tk, int d, int dff, int E, const Ctx& c, cudaStream_t s, void* keep = nullptr);
int launch_tc_down(const void* h, const int32_t* offsets, const void* W2, void* y, int Tk, int d,
                   int dff, int E, const Ctx& c, cudaStream_t s);
// Backward (bf16 activations, fp32 weight gradients).
int dwg_chunks(int T);
// keep == NULL: dh (fp32) to `dh`; else the forward's p and q ([2, Tk, dff]
// bf16) give da = dh p, db = dh q (bf16) to dA, dB directly.
int launch_bwd_dh(const void* dout_perm, const float* w_perm, const int32_t* offsets, const void* W2, float* dh,
                  const void* keep, void* dA, void* dB, int Tk, int d, int dff, int E, const Ctx& c, cudaStream_t s);
int launch_bwd_dsw(const void* x_perm, const float* dh, const int32_t* offsets, const void* W1, const void* W3,
                   void* dA, void* dB, int Tk, int d, int dff, int E, const Ctx& c, cudaStream_t s);
int launch_bwd_dx(const void* dA, const void* dB, const int32_t* offsets, const void* W1, const void* W3,
                  void* dx_perm, int Tk, int d, int dff, int E, const Ctx& c, cudaStream_t s);
int launch_bwd_wgrad(const void* A, const void* B, const int32_t* offsets, float* dW, int M, int N, int Tk,
                     int E, const Ctx& c, cudaStream_t s);
cudaError_t launch_route_bwd(const void* dout, const void* y_perm, const int32_t* slot_pos, const float* w,
                             void* dy_perm, void* dout_perm, float* w_perm, float* dl, int T, int d, int k,
                             const Ctx& c, cudaStream_t s);
cudaError_t launch_dx_gather(const void* dx_perm, const int32_t* slot_pos, const int32_t* idx, const float* dl,
                             const void* Wg, void* dx, int T, int d, int E, int k, const Ctx& c, cudaStream_t s);
cudaError_t launch_dwg(const void* x, const int32_t* idx, const float* dl, float* part, float* dWg, int T, int d,
                       int E, int k, const Ctx& c, cudaStream_t s);
// int8 weight-only path: per-row int8 codes + fp32 scales, bf16 activations.
cudaError_t launch_quantize_int8(const void* W, long long rows, int cols, int8_t* q, float* scale,
                                 const Ctx& c, cudaStream_t s);
int launch_w8_gate_up(const void* x_perm, const int32_t* offsets, const int8_t* W1q, const float* W1s,
                      const int8_t* W3q, const float* W3s, void* h, int Tk, int d, int dff, int E,
                      const Ctx& c, cudaStream_t s);
int launch_w8_down(const void* h, const int32_t* offsets, const int8_t* W2q, const float* W2s, void* y,
                   int Tk, int d, int dff, int E, const Ctx& c, cudaStream_t s);
// The same products beyond the small-batch case: weights widened into tensor
// memory as the MMA's A operand, 224 tokens per tile (ffn_w8_wide.cu).
int launch_w8_wide_gate_up(const void* x_perm, const int32_t* offsets, const int8_t* W1q, const float* W1s,
                           const int8_t* W3q, const float* W3s, void* h, int Tk, int d, int dff, int E,
                           const Ctx& c, cudaStream_t s);
int launch_w8_wide_down(const void* h, const int32_t* offsets, const int8_t* W2q, const float* W2s, void* y,
                        int Tk, int d, int dff, int E, const Ctx& c, cudaStream_t s);

}  // namespace moe
