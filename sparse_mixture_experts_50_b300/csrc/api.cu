// C-ABI entry points of libmoe (declared in include/moe.h).  Host code only:
// argument validation, device selection, workspace layout and the order of
// the kernels of the sparse-MoE layer ("The Evolving Transformer - 05
// Mixtral", sections 03-06):
//   [a0 RMSNorm] -> a1/a2 router -> a3 dispatch (rank, gather) ->
//   a4 gate/up + SwiGLU -> a5 down -> a6 combine [+ residual].
// Everything is enqueued on the caller's stream; no entry point reads a
// device value on the host, so the per-expert counts never leave the GPU.
#include <atomic>
#include <climits>
#include <cmath>
#include <mutex>

#include "moe_internal.cuh"

namespace moe {

// First MOE_E* code any kernel recorded on this device since the last reset.
__device__ int g_status;

namespace {

std::atomic<unsigned long long> g_wait_ns{2000000000ull};

struct DevInfo {
  bool init;
  int num_sms;
  int* status;
};
std::mutex g_mu;
DevInfo g_dev[64];

}  // namespace

int make_ctx(const void* dev_ptr, Ctx* ctx, int* prev_device) {
  *prev_device = -1;
  int dev = -1;
  if (dev_ptr != nullptr) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, dev_ptr) == cudaSuccess &&
        (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged)) {
      dev = a.device;
    } else {
      cudaGetLastError();
    }
  }
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return MOE_ECUDA;
  if (dev < 0) dev = cur;
  if (dev >= 64) return MOE_EUNSUPPORTED;
  if (dev != cur) {
    if (cudaSetDevice(dev) != cudaSuccess) return MOE_ECUDA;
    *prev_device = cur;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo& d = g_dev[dev];
  if (!d.init) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ECUDA;
    void* sp = nullptr;
    if (cudaGetSymbolAddress(&sp, g_status) != cudaSuccess) return MOE_ECUDA;
    d.num_sms = sms;
    d.status = static_cast<int*>(sp);
    d.init = true;
  }
  ctx->device = dev;
  ctx->num_sms = d.num_sms;
  ctx->status = d.status;
  ctx->wait_ns = g_wait_ns.load();
  ctx->max_rows_per_expert = 0;
  return MOE_OK;
}

namespace {

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
inline size_t esize(int dtype) { return dtype == MOE_DTYPE_BF16 ? 2 : 4; }
inline int launch_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ECUDA; }

#define MOE_TRY(expr)          \
  do {                         \
    const int rc_ = (expr);    \
    if (rc_ != MOE_OK) return rc_; \
  } while (0)

int check_dtype(int dtype) { return (dtype == MOE_DTYPE_F32 || dtype == MOE_DTYPE_BF16) ? MOE_OK : MOE_EINVAL; }

// Shape checks shared by the entry points that see tokens.
int check_tokens(int T, int d, int E, int k, int dtype) {
  MOE_TRY(check_dtype(dtype));
  if (T < 0 || d <= 0 || E <= 0 || k <= 0 || k > E) return MOE_EINVAL;
  if (E > 64 || k > 8) return MOE_EUNSUPPORTED;
  if (d % (dtype == MOE_DTYPE_BF16 ? 8 : 4) != 0) return MOE_EUNSUPPORTED;
  if (static_cast<long long>(T) * k > INT_MAX / 2) return MOE_EUNSUPPORTED;
  return MOE_OK;
}

// Shape checks of the expert GEMMs.
int check_ffn(int Tk, int d, int dff, int E, int dtype) {
  MOE_TRY(check_dtype(dtype));
  if (Tk < 0 || d <= 0 || dff <= 0 || E <= 0) return MOE_EINVAL;
  if (E > 64) return MOE_EUNSUPPORTED;
  if (dtype == MOE_DTYPE_BF16) {
    if (d % 64 != 0 || dff % 64 != 0) return MOE_EUNSUPPORTED;
    if (static_cast<long long>(E) * dff > INT_MAX / 2 || static_cast<long long>(E) * d > INT_MAX / 2)
      return MOE_EUNSUPPORTED;
  } else {
    if (d % 4 != 0 || dff % 4 != 0) return MOE_EUNSUPPORTED;
    if (Tk / 64 + E > 65535) return MOE_EUNSUPPORTED;
  }
  return MOE_OK;
}

int ffn_gate_up(const void* x_perm, const int32_t* offsets, const void* W1, const void* W3, void* h, int Tk, int d,
                int dff, int E, int dtype, const Ctx& c, cudaStream_t s, void* keep = nullptr) {
  if (dtype == MOE_DTYPE_BF16) return launch_tc_gate_up(x_perm, offsets, W1, W3, h, Tk, d, dff, E, c, s, keep);
  return launch_rc(launch_ffn_f32_gate_up(static_cast<const float*>(x_perm), offsets, static_cast<const float*>(W1),
                                          static_cast<const float*>(W3), static_cast<float*>(h), Tk, d, dff, E, c, s));
}

int ffn_down(const void* h, const int32_t* offsets, const void* W2, void* y, int Tk, int d, int dff, int E, int dtype,
             const Ctx& c, cudaStream_t s) {
  if (dtype == MOE_DTYPE_BF16) return launch_tc_down(h, offsets, W2, y, Tk, d, dff, E, c, s);
  return launch_rc(launch_ffn_f32_down(static_cast<const float*>(h), offsets, static_cast<const float*>(W2),
                                       static_cast<float*>(y), Tk, d, dff, E, c, s));
}

// int8 expert weights (codes + per-row scales) for the weight-only path.
struct W8Weights {
  const int8_t* q1;
  const float* s1;
  const int8_t* q3;
  const float* s3;
  const int8_t* q2;
  const float* s2;
};

struct WsLayout {
  size_t idx, w, counts, offs, row_src, slot_pos, x_perm, h, y, xn, total;
};

inline size_t al256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

WsLayout ws_layout(int T, int d, int dff, int E, int k, int dtype) {
  const size_t es = esize(dtype);
  const size_t Tk = static_cast<size_t>(T) * k;
  WsLayout L;
  size_t o = 0;
  L.idx = o;       o = al256(o + Tk * 4);
  L.w = o;         o = al256(o + Tk * 4);
  L.counts = o;    o = al256(o + static_cast<size_t>(E) * 4);
  L.offs = o;      o = al256(o + static_cast<size_t>(E + 1) * 4);
  L.row_src = o;   o = al256(o + Tk * 4);
  L.slot_pos = o;  o = al256(o + Tk * 4);
  L.x_perm = o;    o = al256(o + Tk * d * es);
  L.h = o;         o = al256(o + Tk * dff * es);
  L.y = o;         o = al256(o + Tk * d * es);
  L.xn = o;        o = al256(o + static_cast<size_t>(T) * d * es);
  L.total = o;
  return L;
}

// The layer on caller scratch; gamma != NULL selects the block form, w8 !=
// NULL the int8 expert weights (W1, W3, W2 are then unused).
// `events` (optional, 5 caller-created cudaEvent_t) are recorded before the
// router, after dispatch, after gate/up, after down and after combine.
// `keep` (optional, bf16 only) receives p = b silu'(a) and q = silu(a) of the
// gate/up GEMM's a and b in bf16, planes [2, T*k, dff] in the permuted row
// order, for the backward.
int forward_impl(const void* x, const void* gamma, float eps, const void* Wg, const void* W1, const void* W3,
                 const void* W2, void* out, int T, int d, int dff, int E, int k, int dtype, void* ws, size_t ws_bytes,
                 const Ctx& cin, cudaStream_t s, const W8Weights* w8 = nullptr, void* const* events = nullptr,
                 void* keep = nullptr) {
  Ctx c = cin;
  c.max_rows_per_expert = T;  // each token picks an expert at most once
  auto mark = [&](int i) -> int {
    if (events == nullptr || events[i] == nullptr) return MOE_OK;
    return cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) == cudaSuccess ? MOE_OK : MOE_ECUDA;
  };
  const WsLayout L = ws_layout(T, d, dff, E, k, dtype);
  if (ws_bytes < L.total) return MOE_ENOMEM;
  uint8_t* base = static_cast<uint8_t*>(ws);
  int32_t* idx = reinterpret_cast<int32_t*>(base + L.idx);
  float* w = reinterpret_cast<float*>(base + L.w);
  int32_t* counts = reinterpret_cast<int32_t*>(base + L.counts);
  int32_t* offs = reinterpret_cast<int32_t*>(base + L.offs);
  int32_t* row_src = reinterpret_cast<int32_t*>(base + L.row_src);
  int32_t* slot_pos = reinterpret_cast<int32_t*>(base + L.slot_pos);
  void* x_perm = base + L.x_perm;
  void* h = base + L.h;
  void* y = base + L.y;
  const int Tk = T * k;
  const void* xin = x;
  MOE_TRY(mark(0));
  if (gamma != nullptr) {
    void* xn = base + L.xn;
    MOE_TRY(launch_rc(launch_rmsnorm(x, gamma, eps, xn, T, d, dtype, c, s)));
    xin = xn;
  }
  MOE_TRY(launch_rc(launch_router(xin, Wg, T, d, E, k, idx, w, nullptr, dtype, c, s)));
  MOE_TRY(launch_rc(launch_dispatch(idx, Tk, E, k, counts, offs, row_src, slot_pos, c, s)));
  MOE_TRY(launch_rc(launch_gather_rows(xin, row_src, x_perm, T, Tk, static_cast<size_t>(d) * esize(dtype), c, s)));
  MOE_TRY(mark(1));
  if (w8 != nullptr) {
    MOE_TRY(launch_w8_gate_up(x_perm, offs, w8->q1, w8->s1, w8->q3, w8->s3, h, Tk, d, dff, E, c, s));
    MOE_TRY(mark(2));
    MOE_TRY(launch_w8_down(h, offs, w8->q2, w8->s2, y, Tk, d, dff, E, c, s));
  } else {
    MOE_TRY(ffn_gate_up(x_perm, offs, W1, W3, h, Tk, d, dff, E, dtype, c, s, keep));
    MOE_TRY(mark(2));
    MOE_TRY(ffn_down(h, offs, W2, y, Tk, d, dff, E, dtype, c, s));
  }
  MOE_TRY(mark(3));
  MOE_TRY(launch_rc(launch_combine(y, slot_pos, w, gamma != nullptr ? x : nullptr, out, T, d, k, dtype, c, s)));
  MOE_TRY(mark(4));
  return MOE_OK;
}

int check_forward(const void* x, const void* Wg, const void* W1, const void* W3, const void* W2, const void* out,
                  int T, int d, int dff, int E, int k, int dtype) {
  MOE_TRY(check_tokens(T, d, E, k, dtype));
  MOE_TRY(check_ffn(T * k, d, dff, E, dtype));
  if (T == 0) return MOE_OK;
  const void* ptrs[] = {x, Wg, W1, W3, W2, out};
  for (const void* p : ptrs) {
    if (p == nullptr) return MOE_EINVAL;
    if (!aligned(p, 16)) return MOE_EINVAL;
  }
  return MOE_OK;
}

int forward_alloc(const void* x, const void* gamma, float eps, const void* Wg, const void* W1, const void* W3,
                  const void* W2, void* out, int T, int d, int dff, int E, int k, int dtype, cudaStream_t s) {
  MOE_TRY(check_forward(x, Wg, W1, W3, W2, out, T, d, dff, E, k, dtype));
  if (T == 0) return MOE_OK;
  CtxScope scope;
  MOE_TRY(scope.init(out));
  const Ctx& c = scope.ctx();
  const size_t bytes = ws_layout(T, d, dff, E, k, dtype).total;
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, bytes, s) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ENOMEM;
  }
  const int rc = forward_impl(x, gamma, eps, Wg, W1, W3, W2, out, T, d, dff, E, k, dtype, ws, bytes, c, s);
  const cudaError_t fe = cudaFreeAsync(ws, s);
  if (rc != MOE_OK) return rc;
  return fe == cudaSuccess ? MOE_OK : MOE_ECUDA;
}

int check_eps(float eps) { return (std::isfinite(eps) && eps >= 0.0f) ? MOE_OK : MOE_EINVAL; }

int check_w8(const W8Weights& w) {
  const void* ptrs[] = {w.q1, w.s1, w.q3, w.s3, w.q2, w.s2};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned(p, 16)) return MOE_EINVAL;
  return MOE_OK;
}

int forward_w8(const void* x, const void* Wg, const W8Weights& w8, void* out, int T, int d, int dff, int E, int k,
               void* ws, size_t ws_bytes, bool alloc, cudaStream_t s) {
  MOE_TRY(check_tokens(T, d, E, k, MOE_DTYPE_BF16));
  MOE_TRY(check_ffn(T * k, d, dff, E, MOE_DTYPE_BF16));
  if (T == 0) return MOE_OK;
  if (x == nullptr || Wg == nullptr || out == nullptr || !aligned(x, 16) || !aligned(Wg, 16) || !aligned(out, 16))
    return MOE_EINVAL;
  MOE_TRY(check_w8(w8));
  if (!alloc && (ws == nullptr || !aligned(ws, 256))) return MOE_EINVAL;
  CtxScope scope;
  MOE_TRY(scope.init(out));
  const Ctx& c = scope.ctx();
  if (!alloc) {
    return forward_impl(x, nullptr, 0.0f, Wg, nullptr, nullptr, nullptr, out, T, d, dff, E, k, MOE_DTYPE_BF16, ws,
                        ws_bytes, c, s, &w8);
  }
  const size_t bytes = moe_forward_w8_workspace_bytes(T, d, dff, E, k);
  void* buf = nullptr;
  if (cudaMallocAsync(&buf, bytes, s) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ENOMEM;
  }
  const int rc = forward_impl(x, nullptr, 0.0f, Wg, nullptr, nullptr, nullptr, out, T, d, dff, E, k, MOE_DTYPE_BF16,
                              buf, bytes, c, s, &w8);
  const cudaError_t fe = cudaFreeAsync(buf, s);
  if (rc != MOE_OK) return rc;
  return fe == cudaSuccess ? MOE_OK : MOE_ECUDA;
}


// ---- backward ---------------------------------------------------------------
struct BwdLayout {
  size_t dy, dop, wp, dl, dh, dA, dB, dxp, part, total;
};

BwdLayout bwd_layout(int T, int d, int dff, int E, int k) {
  const size_t Tk = static_cast<size_t>(T) * k;
  BwdLayout L;
  size_t o = 0;
  L.dy = o;    o = al256(o + Tk * d * 2);
  L.dop = o;   o = al256(o + Tk * d * 2);
  L.wp = o;    o = al256(o + Tk * 4);
  L.dl = o;    o = al256(o + Tk * 4);
  L.dh = o;    o = al256(o + Tk * dff * 4);
  L.dA = o;    o = al256(o + Tk * dff * 2);
  L.dB = o;    o = al256(o + Tk * dff * 2);
  L.dxp = o;   o = al256(o + Tk * d * 2);
  L.part = o;  o = al256(o + static_cast<size_t>(dwg_chunks(T)) * E * d * 4);
  L.total = o;
  return L;
}

// The backward, B1..B7, on caller scratch; `saved` is the scratch of the
// forward call (moe_forward_ws) on the same x and weights.
int backward_impl(const void* dout, const void* x, const void* Wg, const void* W1, const void* W3, const void* W2,
                  const void* saved, const void* keep, void* dx, float* dWg, float* dW1, float* dW3, float* dW2,
                  int T, int d, int dff, int E, int k, void* ws, const Ctx& c, cudaStream_t s) {
  const WsLayout F = ws_layout(T, d, dff, E, k, MOE_DTYPE_BF16);
  const BwdLayout L = bwd_layout(T, d, dff, E, k);
  const uint8_t* sv = static_cast<const uint8_t*>(saved);
  const int32_t* idx = reinterpret_cast<const int32_t*>(sv + F.idx);
  const float* w = reinterpret_cast<const float*>(sv + F.w);
  const int32_t* offs = reinterpret_cast<const int32_t*>(sv + F.offs);
  const int32_t* slot_pos = reinterpret_cast<const int32_t*>(sv + F.slot_pos);
  const void* x_perm = sv + F.x_perm;
  const void* h = sv + F.h;
  const void* y_perm = sv + F.y;
  uint8_t* b = static_cast<uint8_t*>(ws);
  void* dy = b + L.dy;
  void* dop = b + L.dop;
  float* wp = reinterpret_cast<float*>(b + L.wp);
  float* dl = reinterpret_cast<float*>(b + L.dl);
  void* dA = b + L.dA;
  void* dB = b + L.dB;
  void* dxp = b + L.dxp;
  const int Tk = T * k;
  // B1-B2: expert-output and gate-weight gradients, softmax over the k chosen.
  MOE_TRY(launch_rc(launch_route_bwd(dout, y_perm, slot_pos, w, dy, dop, wp, dl, T, d, k, c, s)));
  // B3: dh = w (dout W2) in fp32 and the SwiGLU derivative -> dA, dB: from
  // the p and q the training forward kept, else with a and b recomputed.
  float* dh = reinterpret_cast<float*>(b + L.dh);
  if (keep != nullptr) {
    MOE_TRY(launch_bwd_dh(dop, wp, offs, W2, nullptr, keep, dA, dB, Tk, d, dff, E, c, s));
  } else {
    MOE_TRY(launch_bwd_dh(dop, wp, offs, W2, dh, nullptr, nullptr, nullptr, Tk, d, dff, E, c, s));
    MOE_TRY(launch_bwd_dsw(x_perm, dh, offs, W1, W3, dA, dB, Tk, d, dff, E, c, s));
  }
  // B4: dx_perm = dA W1 + dB W3.
  MOE_TRY(launch_bwd_dx(dA, dB, offs, W1, W3, dxp, Tk, d, dff, E, c, s));
  // B5: un-permute + router path -> dx.
  MOE_TRY(launch_rc(launch_dx_gather(dxp, slot_pos, idx, dl, Wg, dx, T, d, E, k, c, s)));
  // B6: dWg.
  MOE_TRY(launch_rc(launch_dwg(x, idx, dl, reinterpret_cast<float*>(b + L.part), dWg, T, d, E, k, c, s)));
  // B7: dW2 = dy^T h, dW1 = dA^T x, dW3 = dB^T x per expert, from the
  // token-major rows.
  MOE_TRY(launch_bwd_wgrad(dy, h, offs, dW2, d, dff, Tk, E, c, s));
  MOE_TRY(launch_bwd_wgrad(dA, x_perm, offs, dW1, dff, d, Tk, E, c, s));
  MOE_TRY(launch_bwd_wgrad(dB, x_perm, offs, dW3, dff, d, Tk, E, c, s));
  return MOE_OK;
}

int check_backward(const void* dout, const void* x, const void* Wg, const void* W1, const void* W3, const void* W2,
                   const void* saved, size_t saved_bytes, const void* keep, const void* dx, const float* dWg,
                   const float* dW1, const float* dW3, const float* dW2, int T, int d, int dff, int E, int k) {
  MOE_TRY(check_forward(x, Wg, W1, W3, W2, dx, T, d, dff, E, k, MOE_DTYPE_BF16));
  if (T == 0) return MOE_OK;
  if (static_cast<long long>(E) * dff * d > INT_MAX || static_cast<long long>(T) * k * dff > (1LL << 40))
    return MOE_EUNSUPPORTED;
  const void* ptrs[] = {dout, saved, dWg, dW1, dW3, dW2};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned(p, 16)) return MOE_EINVAL;
  if (!aligned(saved, 256)) return MOE_EINVAL;
  if (keep != nullptr && !aligned(keep, 16)) return MOE_EINVAL;
  if (saved_bytes < ws_layout(T, d, dff, E, k, MOE_DTYPE_BF16).total) return MOE_ENOMEM;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_EINVAL: return "invalid argument";
    case MOE_EUNSUPPORTED: return "unsupported shape or dtype";
    case MOE_ECUDA: return "CUDA call failed";
    case MOE_ETIMEOUT: return "device-side wait timed out";
    case MOE_ENOMEM: return "workspace too small or allocation failed";
    case MOE_EDEVICE: return "device-side bounds check failed";
    default: return "unknown status";
  }
}

int moe_version(void) { return 100; }

int moe_set_wait_limit_ns(long long ns) {
  g_wait_ns.store(ns > 0 ? static_cast<unsigned long long>(ns) : 2000000000ull);
  return MOE_OK;
}

int moe_router_topk(const void* x, const void* Wg, int T, int d, int E, int k, int32_t* topk_idx, float* topk_w,
                    float* logits_opt, int dtype, moe_stream_t stream) {
  MOE_TRY(check_tokens(T, d, E, k, dtype));
  if (T == 0) return MOE_OK;
  if (!x || !Wg || !topk_idx || !topk_w) return MOE_EINVAL;
  if (!aligned(x, 16) || !aligned(Wg, 16) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) ||
      !aligned(logits_opt, 4))
    return MOE_EINVAL;
  CtxScope scope;
  MOE_TRY(scope.init(topk_idx));
  const Ctx& c = scope.ctx();
  return launch_rc(launch_router(x, Wg, T, d, E, k, topk_idx, topk_w, logits_opt, dtype, c, stream));
}

int moe_rmsnorm(const void* x, const void* gamma, float eps, void* xn, int T, int d, int dtype, moe_stream_t stream) {
  MOE_TRY(check_tokens(T, d, 1, 1, dtype));
  MOE_TRY(check_eps(eps));
  if (T == 0) return MOE_OK;
  if (!x || !gamma || !xn || !aligned(x, 16) || !aligned(gamma, 16) || !aligned(xn, 16)) return MOE_EINVAL;
  CtxScope scope;
  MOE_TRY(scope.init(xn));
  const Ctx& c = scope.ctx();
  return launch_rc(launch_rmsnorm(x, gamma, eps, xn, T, d, dtype, c, stream));
}

int moe_permute(const void* x, const int32_t* topk_idx, int T, int d, int E, int k, int32_t* counts,
                int32_t* offsets, int32_t* row_src, int32_t* slot_pos, void* x_perm, int dtype,
                moe_stream_t stream) {
  MOE_TRY(check_tokens(T, d, E, k, dtype));
  if (!counts || !offsets) return MOE_EINVAL;
  if (T > 0 && (!x || !topk_idx || !row_src || !slot_pos || !x_perm)) return MOE_EINVAL;
  if (!aligned(x, 16) || !aligned(x_perm, 16) || !aligned(topk_idx, 4) || !aligned(counts, 4) ||
      !aligned(offsets, 4) || !aligned(row_src, 4) || !aligned(slot_pos, 4))
    return MOE_EINVAL;
  CtxScope scope;
  MOE_TRY(scope.init(offsets));
  const Ctx& c = scope.ctx();
  const int Tk = T * k;
  MOE_TRY(launch_rc(launch_dispatch(topk_idx, Tk, E, k, counts, offsets, row_src, slot_pos, c, stream)));
  if (Tk == 0) return MOE_OK;
  return launch_rc(launch_gather_rows(x, row_src, x_perm, T, Tk, static_cast<size_t>(d) * esize(dtype), c, stream));
}

int moe_gather_rows(const void* src, int src_rows, const int32_t* row_idx, int n_rows, void* dst, size_t row_bytes,
                    moe_stream_t stream) {
  if (src_rows < 0 || n_rows < 0) return MOE_EINVAL;
  if (row_bytes == 0 || row_bytes % 16 != 0 || row_bytes / 16 > INT_MAX) return MOE_EINVAL;
  if (n_rows == 0) return MOE_OK;
  if (!src || !row_idx || !dst || !aligned(src, 16) || !aligned(dst, 16) || !aligned(row_idx, 4)) return MOE_EINVAL;
  if (static_cast<long long>(n_rows) * static_cast<long long>(row_bytes / 16) > (1LL << 40)) return MOE_EUNSUPPORTED;
  CtxScope scope;
  MOE_TRY(scope.init(dst));
  const Ctx& c = scope.ctx();
  return launch_rc(launch_gather_rows(src, row_idx, dst, src_rows, n_rows, row_bytes, c, stream));
}

int moe_expert_gate_up(const void* x_perm, const int32_t* offsets, const void* W1, const void* W3, void* h_perm,
                       int Tk, int d, int dff, int E, int dtype, moe_stream_t stream) {
  MOE_TRY(check_ffn(Tk, d, dff, E, dtype));
  if (Tk == 0) return MOE_OK;
  const void* ptrs[] = {x_perm, offsets, W1, W3, h_perm};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned(p, 16)) return MOE_EINVAL;
  CtxScope scope;
  MOE_TRY(scope.init(h_perm));
  const Ctx& c = scope.ctx();
  return ffn_gate_up(x_perm, offsets, W1, W3, h_perm, Tk, d, dff, E, dtype, c, stream);
}

int moe_expert_down(const void* h_perm, const int32_t* offsets, const void* W2, void* y_perm, int Tk, int d, int dff,
                    int E, int dtype, moe_stream_t stream) {
  MOE_TRY(check_ffn(Tk, d, dff, E, dtype));
  if (Tk == 0) return MOE_OK;
  const void* ptrs[] = {h_perm, offsets, W2, y_perm};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned(p, 16)) return MOE_EINVAL;
  CtxScope scope;
  MOE_TRY(scope.init(y_perm));
  const Ctx& c = scope.ctx();
  return ffn_down(h_perm, offsets, W2, y_perm, Tk, d, dff, E, dtype, c, stream);
}

int moe_expert_ffn_ws(const void* x_perm, const int32_t* offsets, const void* W1, const void* W3, const void* W2,
                      void* h_perm, void* y_perm, int Tk, int d, int dff, int E, int dtype, moe_stream_t stream) {
  MOE_TRY(moe_expert_gate_up(x_perm, offsets, W1, W3, h_perm, Tk, d, dff, E, dtype, stream));
  return moe_expert_down(h_perm, offsets, W2, y_perm, Tk, d, dff, E, dtype, stream);
}

int moe_expert_ffn(const void* x_perm, const int32_t* offsets, const void* W1, const void* W3, const void* W2,
                   void* y_perm, int Tk, int d, int dff, int E, int dtype, moe_stream_t stream) {
  MOE_TRY(check_ffn(Tk, d, dff, E, dtype));
  if (Tk == 0) return MOE_OK;
  const void* ptrs[] = {x_perm, offsets, W1, W3, W2, y_perm};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned(p, 16)) return MOE_EINVAL;
  CtxScope scope;
  MOE_TRY(scope.init(y_perm));
  void* h = nullptr;
  if (cudaMallocAsync(&h, static_cast<size_t>(Tk) * dff * esize(dtype), stream) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ENOMEM;
  }
  const int rc = moe_expert_ffn_ws(x_perm, offsets, W1, W3, W2, h, y_perm, Tk, d, dff, E, dtype, stream);
  const cudaError_t fe = cudaFreeAsync(h, stream);
  if (rc != MOE_OK) return rc;
  return fe == cudaSuccess ? MOE_OK : MOE_ECUDA;
}

int moe_combine(const void* y_perm, const int32_t* slot_pos, const float* topk_w, const void* residual_opt, void* out,
                int T, int d, int k, int dtype, moe_stream_t stream) {
  MOE_TRY(check_tokens(T, d, k, k, dtype));
  if (T == 0) return MOE_OK;
  if (!y_perm || !slot_pos || !topk_w || !out) return MOE_EINVAL;
  if (!aligned(y_perm, 16) || !aligned(out, 16) || !aligned(residual_opt, 16) || !aligned(slot_pos, 4) ||
      !aligned(topk_w, 4))
    return MOE_EINVAL;
  CtxScope scope;
  MOE_TRY(scope.init(out));
  const Ctx& c = scope.ctx();
  return launch_rc(launch_combine(y_perm, slot_pos, topk_w, residual_opt, out, T, d, k, dtype, c, stream));
}

int moe_forward_workspace_offsets(int T, int d, int dff, int E, int k, int dtype, size_t* offs) {
  MOE_TRY(check_tokens(T, d, E, k, dtype));
  if (dff <= 0) return MOE_EINVAL;
  if (offs == nullptr) return MOE_EINVAL;
  const WsLayout L = ws_layout(T, d, dff, E, k, dtype);
  const size_t v[11] = {L.idx, L.w, L.counts, L.offs, L.row_src, L.slot_pos, L.x_perm, L.h, L.y, L.xn, L.total};
  for (int i = 0; i < 11; ++i) offs[i] = v[i];
  return MOE_OK;
}

size_t moe_workspace_bytes(int T, int d, int dff, int E, int k, int dtype) {
  if (check_tokens(T, d, E, k, dtype) != MOE_OK || dff <= 0) return 0;
  return ws_layout(T, d, dff, E, k, dtype).total;
}

size_t moe_forward_w8_workspace_bytes(int T, int d, int dff, int E, int k) {
  if (check_tokens(T, d, E, k, MOE_DTYPE_BF16) != MOE_OK || dff <= 0) return 0;
  return ws_layout(T, d, dff, E, k, MOE_DTYPE_BF16).total;
}

int moe_forward_ws(const void* x, const void* Wg, const void* W1, const void* W3, const void* W2, void* out, int T,
                   int d, int dff, int E, int k, int dtype, void* workspace, size_t workspace_bytes,
                   moe_stream_t stream) {
  MOE_TRY(check_forward(x, Wg, W1, W3, W2, out, T, d, dff, E, k, dtype));
  if (T == 0) return MOE_OK;
  if (workspace == nullptr || !aligned(workspace, 256)) return MOE_EINVAL;
  CtxScope scope;
  MOE_TRY(scope.init(out));
  const Ctx& c = scope.ctx();
  return forward_impl(x, nullptr, 0.0f, Wg, W1, W3, W2, out, T, d, dff, E, k, dtype, workspace, workspace_bytes, c,
                      stream);
}

int moe_forward_train_ws(const void* x, const void* Wg, const void* W1, const void* W3, const void* W2, void* out,
                         void* keep, int T, int d, int dff, int E, int k, void* workspace,
                         size_t workspace_bytes, moe_stream_t stream) {
  MOE_TRY(check_forward(x, Wg, W1, W3, W2, out, T, d, dff, E, k, MOE_DTYPE_BF16));
  if (T == 0) return MOE_OK;
  if (workspace == nullptr || !aligned(workspace, 256)) return MOE_EINVAL;
  if (keep == nullptr || !aligned(keep, 16)) return MOE_EINVAL;
  CtxScope scope;
  MOE_TRY(scope.init(out));
  const Ctx& c = scope.ctx();
  return forward_impl(x, nullptr, 0.0f, Wg, W1, W3, W2, out, T, d, dff, E, k, MOE_DTYPE_BF16, workspace,
                      workspace_bytes, c, stream, nullptr, nullptr, keep);
}

int moe_forward(const void* x, const void* Wg, const void* W1, const void* W3, const void* W2, void* out, int T, int d,
                int dff, int E, int k, moe_stream_t stream) {
  return forward_alloc(x, nullptr, 0.0f, Wg, W1, W3, W2, out, T, d, dff, E, k, MOE_DTYPE_BF16, stream);
}

int moe_forward_f32(const void* x, const void* Wg, const void* W1, const void* W3, const void* W2, void* out, int T,
                    int d, int dff, int E, int k, moe_stream_t stream) {
  return forward_alloc(x, nullptr, 0.0f, Wg, W1, W3, W2, out, T, d, dff, E, k, MOE_DTYPE_F32, stream);
}

int moe_block_forward_ws(const void* x, const void* gamma, float eps, const void* Wg, const void* W1, const void* W3,
                         const void* W2, void* out, int T, int d, int dff, int E, int k, int dtype, void* workspace,
                         size_t workspace_bytes, moe_stream_t stream) {
  MOE_TRY(check_forward(x, Wg, W1, W3, W2, out, T, d, dff, E, k, dtype));
  MOE_TRY(check_eps(eps));
  if (T == 0) return MOE_OK;
  if (gamma == nullptr || !aligned(gamma, 16)) return MOE_EINVAL;
  if (workspace == nullptr || !aligned(workspace, 256)) return MOE_EINVAL;
  CtxScope scope;
  MOE_TRY(scope.init(out));
  const Ctx& c = scope.ctx();
  return forward_impl(x, gamma, eps, Wg, W1, W3, W2, out, T, d, dff, E, k, dtype, workspace, workspace_bytes, c,
                      stream);
}

int moe_block_forward(const void* x, const void* gamma, float eps, const void* Wg, const void* W1, const void* W3,
                      const void* W2, void* out, int T, int d, int dff, int E, int k, moe_stream_t stream) {
  MOE_TRY(check_eps(eps));
  if (T > 0 && (gamma == nullptr || !aligned(gamma, 16))) return MOE_EINVAL;
  return forward_alloc(x, gamma, eps, Wg, W1, W3, W2, out, T, d, dff, E, k, MOE_DTYPE_BF16, stream);
}

size_t moe_forward_host_workspace_bytes(int T, int d, int dff, int E, int k, int dtype) {
  const size_t base = moe_workspace_bytes(T, d, dff, E, k, dtype);
  if (base == 0) return 0;
  const size_t act = al256(static_cast<size_t>(T) * d * esize(dtype));
  return base + 2 * act;
}

int moe_forward_host(const void* x_host, const void* Wg, const void* W1, const void* W3, const void* W2,
                     void* out_host, int T, int d, int dff, int E, int k, int dtype, void* workspace,
                     size_t workspace_bytes, moe_stream_t stream) {
  MOE_TRY(check_forward(x_host, Wg, W1, W3, W2, out_host, T, d, dff, E, k, dtype));
  if (T == 0) return MOE_OK;
  if (workspace == nullptr || !aligned(workspace, 256)) return MOE_EINVAL;
  const size_t need = moe_forward_host_workspace_bytes(T, d, dff, E, k, dtype);
  if (workspace_bytes < need) return MOE_ENOMEM;
  CtxScope scope;
  MOE_TRY(scope.init(Wg));
  const Ctx& c = scope.ctx();
  const size_t base = moe_workspace_bytes(T, d, dff, E, k, dtype);
  const size_t act_bytes = static_cast<size_t>(T) * d * esize(dtype);
  uint8_t* x_dev = static_cast<uint8_t*>(workspace) + base;
  uint8_t* out_dev = x_dev + al256(act_bytes);
  if (cudaMemcpyAsync(x_dev, x_host, act_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess) return MOE_ECUDA;
  MOE_TRY(forward_impl(x_dev, nullptr, 0.0f, Wg, W1, W3, W2, out_dev, T, d, dff, E, k, dtype, workspace, base, c,
                       stream));
  if (cudaMemcpyAsync(out_host, out_dev, act_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return MOE_ECUDA;
  return cudaStreamSynchronize(stream) == cudaSuccess ? MOE_OK : MOE_ECUDA;
}

int moe_forward_ex(const void* x, const void* gamma_opt, float eps, const void* Wg, const void* W1, const void* W3,
                   const void* W2, const int8_t* W1q, const float* W1s, const int8_t* W3q, const float* W3s,
                   const int8_t* W2q, const float* W2s, void* out, int T, int d, int dff, int E, int k, int dtype,
                   void* workspace, size_t workspace_bytes, void* const* events, moe_stream_t stream) {
  const bool w8 = W1q != nullptr;
  if (w8 && dtype != MOE_DTYPE_BF16) return MOE_EUNSUPPORTED;
  const W8Weights q{W1q, W1s, W3q, W3s, W2q, W2s};
  // The shape and pointer checks of the plain layer; with int8 weights the
  // bf16 ones are not used (Wg stands in for them in the null check).
  MOE_TRY(check_forward(x, Wg, w8 ? Wg : W1, w8 ? Wg : W3, w8 ? Wg : W2, out, T, d, dff, E, k, dtype));
  if (gamma_opt != nullptr) MOE_TRY(check_eps(eps));
  if (T == 0) return MOE_OK;
  if (w8) MOE_TRY(check_w8(q));
  if (gamma_opt != nullptr && !aligned(gamma_opt, 16)) return MOE_EINVAL;
  if (workspace == nullptr || !aligned(workspace, 256)) return MOE_EINVAL;
  CtxScope scope;
  MOE_TRY(scope.init(out));
  const Ctx& c = scope.ctx();
  return forward_impl(x, gamma_opt, eps, Wg, W1, W3, W2, out, T, d, dff, E, k, dtype, workspace, workspace_bytes, c,
                      stream, w8 ? &q : nullptr, events);
}

int moe_quantize_int8(const void* W, int rows, int cols, int8_t* q, float* scale, moe_stream_t stream) {
  if (rows < 0 || cols <= 0) return MOE_EINVAL;
  if (cols % 8 != 0) return MOE_EUNSUPPORTED;
  if (rows == 0) return MOE_OK;
  if (!W || !q || !scale || !aligned(W, 16) || !aligned(q, 16) || !aligned(scale, 4)) return MOE_EINVAL;
  CtxScope scope;
  MOE_TRY(scope.init(q));
  const Ctx& c = scope.ctx();
  return launch_rc(launch_quantize_int8(W, rows, cols, q, scale, c, stream));
}

int moe_expert_gate_up_w8(const void* x_perm, const int32_t* offsets, const int8_t* W1q, const float* W1s,
                          const int8_t* W3q, const float* W3s, void* h_perm, int Tk, int d, int dff, int E,
                          moe_stream_t stream) {
  MOE_TRY(check_ffn(Tk, d, dff, E, MOE_DTYPE_BF16));
  if (Tk == 0) return MOE_OK;
  const void* ptrs[] = {x_perm, offsets, W1q, W1s, W3q, W3s, h_perm};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned(p, 16)) return MOE_EINVAL;
  CtxScope scope;
  MOE_TRY(scope.init(h_perm));
  const Ctx& c = scope.ctx();
  return launch_w8_gate_up(x_perm, offsets, W1q, W1s, W3q, W3s, h_perm, Tk, d, dff, E, c, stream);
}

int moe_expert_down_w8(const void* h_perm, const int32_t* offsets, const int8_t* W2q, const float* W2s, void* y_perm,
                       int Tk, int d, int dff, int E, moe_stream_t stream) {
  MOE_TRY(check_ffn(Tk, d, dff, E, MOE_DTYPE_BF16));
  if (Tk == 0) return MOE_OK;
  const void* ptrs[] = {h_perm, offsets, W2q, W2s, y_perm};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned(p, 16)) return MOE_EINVAL;
  CtxScope scope;
  MOE_TRY(scope.init(y_perm));
  const Ctx& c = scope.ctx();
  return launch_w8_down(h_perm, offsets, W2q, W2s, y_perm, Tk, d, dff, E, c, stream);
}

int moe_forward_w8_ws(const void* x, const void* Wg, const int8_t* W1q, const float* W1s, const int8_t* W3q,
                      const float* W3s, const int8_t* W2q, const float* W2s, void* out, int T, int d, int dff, int E,
                      int k, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  const W8Weights w8{W1q, W1s, W3q, W3s, W2q, W2s};
  return forward_w8(x, Wg, w8, out, T, d, dff, E, k, workspace, workspace_bytes, false, stream);
}

int moe_forward_w8(const void* x, const void* Wg, const int8_t* W1q, const float* W1s, const int8_t* W3q,
                   const float* W3s, const int8_t* W2q, const float* W2s, void* out, int T, int d, int dff, int E,
                   int k, moe_stream_t stream) {
  const W8Weights w8{W1q, W1s, W3q, W3s, W2q, W2s};
  return forward_w8(x, Wg, w8, out, T, d, dff, E, k, nullptr, 0, true, stream);
}

size_t moe_backward_workspace_bytes(int T, int d, int dff, int E, int k) {
  if (check_tokens(T, d, E, k, MOE_DTYPE_BF16) != MOE_OK || dff <= 0) return 0;
  return bwd_layout(T, d, dff, E, k).total;
}

int moe_backward_ws(const void* dout, const void* x, const void* Wg, const void* W1, const void* W3, const void* W2,
                    const void* saved, size_t saved_bytes, const void* keep, void* dx, float* dWg, float* dW1,
                    float* dW3, float* dW2, int T, int d, int dff, int E, int k, void* workspace,
                    size_t workspace_bytes, moe_stream_t stream) {
  MOE_TRY(check_backward(dout, x, Wg, W1, W3, W2, saved, saved_bytes, keep, dx, dWg, dW1, dW3, dW2, T, d, dff, E,
                         k));
  if (T == 0) return MOE_OK;
  if (workspace == nullptr || !aligned(workspace, 256)) return MOE_EINVAL;
  if (workspace_bytes < bwd_layout(T, d, dff, E, k).total) return MOE_ENOMEM;
  CtxScope scope;
  MOE_TRY(scope.init(dx));
  const Ctx& c = scope.ctx();
  return backward_impl(dout, x, Wg, W1, W3, W2, saved, keep, dx, dWg, dW1, dW3, dW2, T, d, dff, E, k, workspace,
                       c, stream);
}

int moe_backward(const void* dout, const void* x, const void* Wg, const void* W1, const void* W3, const void* W2,
                 const void* saved, size_t saved_bytes, const void* keep, void* dx, float* dWg, float* dW1,
                 float* dW3, float* dW2, int T, int d, int dff, int E, int k, moe_stream_t stream) {
  MOE_TRY(check_backward(dout, x, Wg, W1, W3, W2, saved, saved_bytes, keep, dx, dWg, dW1, dW3, dW2, T, d, dff, E,
                         k));
  if (T == 0) return MOE_OK;
  CtxScope scope;
  MOE_TRY(scope.init(dx));
  const Ctx& c = scope.ctx();
  const size_t bytes = bwd_layout(T, d, dff, E, k).total;
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, bytes, stream) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ENOMEM;
  }
  const int rc =
      backward_impl(dout, x, Wg, W1, W3, W2, saved, keep, dx, dWg, dW1, dW3, dW2, T, d, dff, E, k, ws, c, stream);
  const cudaError_t fe = cudaFreeAsync(ws, stream);
  if (rc != MOE_OK) return rc;
  return fe == cudaSuccess ? MOE_OK : MOE_ECUDA;
}

int moe_get_device_status(moe_stream_t stream, int* status, int reset) {
  if (status == nullptr) return MOE_EINVAL;
  int dev = 0;
  if (cudaStreamGetDevice(stream, &dev) != cudaSuccess) return MOE_ECUDA;
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return MOE_ECUDA;
  if (dev != cur && cudaSetDevice(dev) != cudaSuccess) return MOE_ECUDA;
  int rc = MOE_OK;
  int v = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess || cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) {
    rc = MOE_ECUDA;
  } else if (reset) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_status, &z, sizeof(int)) != cudaSuccess) rc = MOE_ECUDA;
  }
  if (dev != cur) cudaSetDevice(cur);  // the caller's current device again
  if (rc == MOE_OK) *status = v;
  return rc;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// moe_forward_noalloc: the bf16 layer for callers that must not allocate
// device memory while they run (for example an application whose memory
// manager owns the whole device budget and forbids allocation after start-up,
// or a latency-critical loop where a cudaMalloc could synchronise the device).
// Its scratch is this file-scope array: it is part of the library's device
// image, so every GPU that loads the library holds it until the process
// exits, and all calls share it.
namespace moe {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current (in host code the symbol's name is only a host-side handle).
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

int noalloc_scratch(int device, void** ptr) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[device] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ECUDA;
    }
    g_noalloc_ptr[device] = p;
  }
  *ptr = g_noalloc_ptr[device];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_forward_noalloc(const void* x, const void* Wg, const void* W1, const void* W3, const void* W2,
                                   void* out, int T, int d, int dff, int E, int k, moe_stream_t stream) {
  MOE_TRY(check_forward(x, Wg, W1, W3, W2, out, T, d, dff, E, k, MOE_DTYPE_BF16));
  if (T == 0) return MOE_OK;
  const size_t need = ws_layout(T, d, dff, E, k, MOE_DTYPE_BF16).total;
  if (need > MOE_NOALLOC_SCRATCH_BYTES) return MOE_ENOMEM;
  CtxScope scope;
  MOE_TRY(scope.init(out));
  const Ctx& c = scope.ctx();
  void* scratch = nullptr;
  MOE_TRY(noalloc_scratch(c.device, &scratch));
  // Every step writes all the scratch it later reads (indices, weights,
  // permuted rows, h, y), so nothing left by an earlier call is used and
  // nothing needs clearing.
  return forward_impl(x, nullptr, 0.0f, Wg, W1, W3, W2, out, T, d, dff, E, k, MOE_DTYPE_BF16, scratch,
                      MOE_NOALLOC_SCRATCH_BYTES, c, stream);
}
