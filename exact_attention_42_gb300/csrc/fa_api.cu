// The C entry points of libfa.so (declared in include/fa.h): argument
// checks, per-device set-up and dispatch to the kernels' launch functions.
// Every check here happens before anything is enqueued, so an argument error
// leaves the outputs untouched.

#include <cuda_runtime.h>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <memory>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace fa {

struct DeviceInfo {
  bool ok = false;
  bool supported = false;
  int sms = 0;
};

// Test hook state (process-wide): see fa_debug_fault_injection and
// fa_debug_soft_exp.
static std::atomic<int> g_fault_mode{0};
static std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitLimitNs};
static std::atomic<int> g_soft_exp{0};
static std::atomic<int> g_fwd_pair{0};

static DeviceInfo g_dev[kMaxDevicesDecode];
static std::mutex g_dev_mutex;

// Launch settings of the current device: FA_ERR_UNSUPPORTED unless it is sm_103.
static fa_status launch_env(LaunchEnv* env) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevicesDecode) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& di = g_dev[dev];
  if (!di.ok) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    di.supported = (major == 10 && minor == 3);
    di.sms = sms;
    di.ok = true;
  }
  if (!di.supported) return FA_ERR_UNSUPPORTED;
  env->device = dev;
  env->sms = di.sms;
  env->wait_limit_ns = g_wait_limit_ns.load();
  env->fault_mode = g_fault_mode.load();
  env->soft_exp = g_soft_exp.load();
  env->fwd_pair = g_fwd_pair.load();
  return FA_OK;
}

fa_status check_device() {
  LaunchEnv env;
  return launch_env(&env);
}

}  // namespace fa

extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                 int Nk, int d, float scale, int causal, const int32_t* cu_seqlens, cudaStream_t stream) {
  if (B < 0 || Hq < 0 || Hkv < 1 || Nq < 0 || Nk < 0) return FA_ERR_SHAPE;
  if (Hq % Hkv != 0) return FA_ERR_SHAPE;
  if (cu_seqlens != nullptr && Nq != Nk) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_VALUE;
  if (B == 0 || Hq == 0 || Nq == 0) return FA_OK;
  if (q == nullptr || o == nullptr || lse == nullptr) return FA_ERR_NULL;
  if (Nk > 0 && (k == nullptr || v == nullptr)) return FA_ERR_NULL;
  auto mis16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
  if (mis16(q) || mis16(o) || (Nk > 0 && (mis16(k) || mis16(v)))) return FA_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_ALIGN;
  if (cu_seqlens != nullptr && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return FA_ERR_ALIGN;
  // Row and element offsets are 64-bit; the tensor-map row count must fit 32 bits.
  if (cu_seqlens == nullptr && static_cast<long long>(B) * Hq > 0x7fffffffLL) return FA_ERR_SHAPE;
  fa::LaunchEnv env;
  const fa_status st = fa::launch_env(&env);
  if (st != FA_OK) return st;
  return fa::launch_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, cu_seqlens, stream, env);
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_NULL: return "FA_ERR_NULL: a required pointer is NULL";
    case FA_ERR_SHAPE: return "FA_ERR_SHAPE: invalid sizes";
    case FA_ERR_ALIGN: return "FA_ERR_ALIGN: misaligned pointer";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: head dim or device not supported";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA call failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel wait timed out";
    case FA_ERR_VALUE: return "FA_ERR_VALUE: scale must be finite and positive";
  }
  return "unknown fa_status";
}

fa_status fa_device_status(int* bits) {
  if (bits == nullptr) return FA_ERR_NULL;
  // Every stream of the device must be idle first: the word reads and clears
  // below go through the legacy stream, which does not wait for non-blocking
  // streams, and a kernel still running there could set a bit between them.
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
  int v = fa::fwd_status_and_clear();
  if (v < 0) return FA_ERR_CUDA;
  const int dv = fa::decode_status_and_clear();
  if (dv < 0) return FA_ERR_CUDA;
  if (dv) v |= 1 << 8;  // the split-KV kernel gave up on a wait
  const int bv = fa::bwd_status_and_clear();
  if (bv < 0) return FA_ERR_CUDA;
  v |= bv << 9;  // backward kernels: roles 0-2 (dQ) and 4-6 (dK/dV)
  const int qv = fa::quant_status_and_clear();
  if (qv < 0) return FA_ERR_CUDA;
  if (qv) v |= 1 << 16;  // the one-launch quantizer gave up waiting for its copies
  *bits = v;
  return v ? FA_ERR_TIMEOUT : FA_OK;
}

fa_status fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                    int Nk, int d, float scale, int causal, cudaStream_t stream) {
  if (B < 0 || Hq < 0 || Hkv < 1 || Nq < 0 || Nk < 0) return FA_ERR_SHAPE;
  if (Hq % Hkv != 0) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_VALUE;
  if (B == 0 || Hq == 0 || Nq == 0) return FA_OK;
  if (!fa::decode_supported(B, Hq, Hkv, Nq, Nk, d, nullptr)) return FA_ERR_UNSUPPORTED;
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || lse == nullptr) return FA_ERR_NULL;
  auto mis16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
  if (mis16(q) || mis16(k) || mis16(v) || mis16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_ALIGN;
  fa::LaunchEnv env;
  const fa_status st = fa::launch_env(&env);
  if (st != FA_OK) return st;
  return fa::launch_decode(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, stream, env.sms,
                           env.wait_limit_ns, env.fault_mode);
}

int fa_decode_smem_bytes(int d) { return fa::decode_smem_bytes(d); }

fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_descale,
                     const float* k_descale, const float* v_descale, void* o, float* lse, int B, int Hq, int Hkv,
                     int Nq, int Nk, int d, float scale, int causal, const int32_t* cu_seqlens, cudaStream_t stream) {
  if (B < 0 || Hq < 0 || Hkv < 1 || Nq < 0 || Nk < 0) return FA_ERR_SHAPE;
  if (Hq % Hkv != 0) return FA_ERR_SHAPE;
  if (cu_seqlens != nullptr && Nq != Nk) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (Nk % 16 != 0) return FA_ERR_SHAPE;  // rows of V^T are Nk bytes: a multiple of 16
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_VALUE;
  if (B == 0 || Hq == 0 || Nq == 0) return FA_OK;
  if (q8 == nullptr || q_descale == nullptr || o == nullptr || lse == nullptr) return FA_ERR_NULL;
  if (Nk > 0 && (k8 == nullptr || vt8 == nullptr || k_descale == nullptr || v_descale == nullptr))
    return FA_ERR_NULL;
  auto mis = [](const void* ptr, unsigned a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0; };
  if (mis(q8, 16) || mis(o, 16) || (Nk > 0 && (mis(k8, 16) || mis(vt8, 16)))) return FA_ERR_ALIGN;
  if (mis(lse, 4) || mis(q_descale, 4) || (Nk > 0 && (mis(k_descale, 4) || mis(v_descale, 4)))) return FA_ERR_ALIGN;
  if (cu_seqlens != nullptr && mis(cu_seqlens, 4)) return FA_ERR_ALIGN;
  if (cu_seqlens == nullptr && static_cast<long long>(B) * Hq > 0x7fffffffLL) return FA_ERR_SHAPE;
  fa::LaunchEnv env;
  const fa_status st = fa::launch_env(&env);
  if (st != FA_OK) return st;
  return fa::launch_fwd_fp8(q8, k8, vt8, q_descale, k_descale, v_descale, o, lse, B, Hq, Hkv, Nq, Nk, d, scale,
                            causal, cu_seqlens, stream, env);
}

fa_status fa_fp8_quantize(const void* x, void* x8, float* descale, int B, int H, int N, int d, int transpose,
                          const int8_t* signs, cudaStream_t stream) {
  if (B < 0 || H < 0 || N < 0) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (transpose && N % 16 != 0) return FA_ERR_SHAPE;  // rows of the transpose are N bytes
  if (B == 0 || H == 0) return FA_OK;
  if (static_cast<long long>(B) * H > 0x7fffffffLL) return FA_ERR_SHAPE;
  if (descale == nullptr) return FA_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(descale) & 3u) != 0) return FA_ERR_ALIGN;
  const long long blocks = static_cast<long long>(B) * H * ((N + 63) / 64);
  if (blocks > 0x7fffffffLL) return FA_ERR_SHAPE;
  if (N > 0) {
    if (x == nullptr || x8 == nullptr) return FA_ERR_NULL;
    auto mis16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
    if (mis16(x) || mis16(x8)) return FA_ERR_ALIGN;
  }
  fa::LaunchEnv env;
  const fa_status st = fa::launch_env(&env);
  if (st != FA_OK) return st;
  return fa::launch_fp8_quantize(x, x8, descale, B, H, N, d, transpose, signs, stream, env);
}

int fa_bwd_smem_bytes(int d) { return fa::bwd_smem_bytes(d); }

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, float* delta, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                 float scale, int causal, const int32_t* cu_seqlens, cudaStream_t stream) {
  if (B < 0 || Hq < 0 || Hkv < 1 || Nq < 0 || Nk < 0) return FA_ERR_SHAPE;
  if (Hq % Hkv != 0) return FA_ERR_SHAPE;
  if (cu_seqlens != nullptr && Nq != Nk) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_VALUE;
  if (B == 0 || Hq == 0 || Nq == 0) return FA_OK;
  if (q == nullptr || o == nullptr || dout == nullptr || lse == nullptr || dq == nullptr || delta == nullptr)
    return FA_ERR_NULL;
  if (Nk > 0 && (k == nullptr || v == nullptr || dk == nullptr || dv == nullptr)) return FA_ERR_NULL;
  auto mis16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
  if (mis16(q) || mis16(o) || mis16(dout) || mis16(dq)) return FA_ERR_ALIGN;
  if (Nk > 0 && (mis16(k) || mis16(v) || mis16(dk) || mis16(dv))) return FA_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0 || (reinterpret_cast<uintptr_t>(delta) & 3u) != 0)
    return FA_ERR_ALIGN;
  if (cu_seqlens != nullptr && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return FA_ERR_ALIGN;
  if (cu_seqlens == nullptr && static_cast<long long>(B) * Hq > 0x7fffffffLL) return FA_ERR_SHAPE;
  fa::LaunchEnv env;
  const fa_status st = fa::launch_env(&env);
  if (st != FA_OK) return st;
  return fa::launch_bwd(q, k, v, o, dout, lse, dq, dk, dv, delta, B, Hq, Hkv, Nq, Nk, d, scale, causal, cu_seqlens,
                        stream, env.sms, env.wait_limit_ns, env.fault_mode);
}

fa_status fa_debug_fault_injection(int mode, double wait_limit_seconds) {
  if (mode < 0 || mode >= fa::kFaultModes) return FA_ERR_VALUE;
  if (!(wait_limit_seconds <= 10.0)) return FA_ERR_VALUE;  // also rejects NaN
  const unsigned long long ns = wait_limit_seconds > 0.0
                                    ? static_cast<unsigned long long>(wait_limit_seconds * 1e9)
                                    : fa::kDefaultWaitLimitNs;
  fa::g_wait_limit_ns.store(ns);
  fa::g_fault_mode.store(mode);
  return FA_OK;
}

fa_status fa_debug_soft_exp(int on) {
  if (on != 0 && on != 1) return FA_ERR_VALUE;
  fa::g_soft_exp.store(on);
  return FA_OK;
}

fa_status fa_debug_fwd_pair(int on) {
  if (on != 0 && on != 1) return FA_ERR_VALUE;
  fa::g_fwd_pair.store(on);
  return FA_OK;
}

fa_status fa_debug_schedule(int kernel, int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, int workers,
                             int32_t* start, int32_t* units, int capacity, int* table_workers) {
  if (start == nullptr || units == nullptr || table_workers == nullptr) return FA_ERR_NULL;
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Nq < 0 || Nk < 0 || workers < 1) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_SHAPE;
  std::unique_ptr<fa::SchedTable> sc(new fa::SchedTable);
  bool ok = false;
  if (kernel == 0 || kernel == 1)
    ok = fa::fwd_schedule_for(kernel, B, Hq, Hkv, Nq, Nk, d, causal, workers, sc.get());
  else if (kernel == 2 || kernel == 3)
    ok = fa::bwd_schedule_for(kernel - 2, B, Hq, Hkv, Nq, Nk, d, causal, workers, sc.get());
  else
    return FA_ERR_VALUE;
  if (!ok) return FA_ERR_SHAPE;
  *table_workers = sc->workers;
  if (sc->workers == 0) return FA_OK;
  const int n = sc->start[sc->workers];
  if (capacity < n) return FA_ERR_SHAPE;
  for (int w = 0; w <= sc->workers; ++w) start[w] = sc->start[w];
  for (int i = 0; i < n; ++i) units[i] = sc->unit[i];
  return FA_OK;
}

fa_status fa_debug_exp2_soft(const float* x, float* y, int n, cudaStream_t stream) {
  if (n < 0) return FA_ERR_SHAPE;
  if (n == 0) return FA_OK;
  if (x == nullptr || y == nullptr) return FA_ERR_NULL;
  return fa::launch_exp2_soft(x, y, n, stream);
}

int fa_fwd_smem_bytes(int d) { return fa::fwd_smem_bytes(d); }

int fa_fwd_threads(void) { return fa::fwd_threads(); }

}  // extern "C"
