// fa_fwd_host: the forward from host buffers (declared in include/fa.h).
//
// The problem is cut into pieces: a (batch, key/value head range) slice of a
// dense problem with its query heads, or the whole packed batch.  Each
// piece's host-to-device copies run on a copy-in stream, its kernel on the
// caller's stream and its device-to-host copies on a copy-out stream, with
// events between them, so that the copies of one piece overlap the kernel
// and the copies of others.  Pieces of a dense problem are contiguous in
// every tensor, so each copy is one cudaMemcpyAsync.  The two copy streams
// are created once per device and kept for the life of the process; the
// events are created per call.

#include <cuda_runtime.h>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "fa.h"
#include "fa_internal.h"

namespace fa {
namespace {

struct CopyStreams {
  cudaStream_t in = nullptr;
  cudaStream_t out = nullptr;
};

std::mutex g_copy_mu;
CopyStreams g_copy[kMaxDevicesDecode];

fa_status copy_streams(CopyStreams* cs) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesDecode) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_copy_mu);
  CopyStreams& c = g_copy[dev];
  if (c.in == nullptr) {
    if (cudaStreamCreateWithFlags(&c.in, cudaStreamNonBlocking) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaStreamCreateWithFlags(&c.out, cudaStreamNonBlocking) != cudaSuccess) {
      cudaStreamDestroy(c.in);
      c.in = nullptr;
      return FA_ERR_CUDA;
    }
  }
  *cs = c;
  return FA_OK;
}

// Events of one call; destroyed when the call returns (CUDA releases an
// event still pending once it completes).
struct Events {
  std::vector<cudaEvent_t> ev;
  ~Events() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
  }
  cudaEvent_t make() {
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    ev.push_back(e);
    return e;
  }
};

bool copy(void* dst, const void* src, size_t bytes, cudaMemcpyKind kind, cudaStream_t s) {
  return bytes == 0 || cudaMemcpyAsync(dst, src, bytes, kind, s) == cudaSuccess;
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h,
                                 void* q_d, void* k_d, void* v_d, void* o_d, float* lse_d, int B, int Hq, int Hkv,
                                 int Nq, int Nk, int d, float scale, int causal, const int32_t* cu_seqlens_h,
                                 int32_t* cu_seqlens_d, int pieces, cudaStream_t stream) {
  if (B < 0 || Hq < 0 || Hkv < 1 || Nq < 0 || Nk < 0 || pieces < 1) return FA_ERR_SHAPE;
  if (Hq % Hkv != 0) return FA_ERR_SHAPE;
  const bool packed = cu_seqlens_h != nullptr;
  if (packed && Nq != Nk) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA_ERR_VALUE;
  if (B == 0 || Hq == 0 || Nq == 0) return FA_OK;
  if (q_h == nullptr || o_h == nullptr || lse_h == nullptr || q_d == nullptr || o_d == nullptr || lse_d == nullptr)
    return FA_ERR_NULL;
  if (Nk > 0 && (k_h == nullptr || v_h == nullptr || k_d == nullptr || v_d == nullptr)) return FA_ERR_NULL;
  if (packed && cu_seqlens_d == nullptr) return FA_ERR_NULL;
  auto mis16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
  if (mis16(q_d) || mis16(o_d) || (Nk > 0 && (mis16(k_d) || mis16(v_d)))) return FA_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(lse_d) & 3u) != 0) return FA_ERR_ALIGN;
  if (packed && (reinterpret_cast<uintptr_t>(cu_seqlens_d) & 3u) != 0) return FA_ERR_ALIGN;
  if (!packed && static_cast<long long>(B) * Hq > 0x7fffffffLL) return FA_ERR_SHAPE;

  fa_status st = fa::check_device();
  if (st != FA_OK) return st;
  fa::CopyStreams cs;
  st = fa::copy_streams(&cs);
  if (st != FA_OK) return st;
  fa::Events events;
  // The device buffers may still be in use by earlier work on `stream`.
  cudaEvent_t start = events.make();
  if (start == nullptr || cudaEventRecord(start, stream) != cudaSuccess ||
      cudaStreamWaitEvent(cs.in, start, 0) != cudaSuccess || cudaStreamWaitEvent(cs.out, start, 0) != cudaSuccess)
    return FA_ERR_CUDA;

  // From here on an error still orders later work on `stream` after every
  // copy already issued on the copy streams (best effort: these calls report
  // nothing further), so the caller may reuse its buffers once `stream` is done.
  auto fail = [&](fa_status code) {
    cudaEvent_t in_end = events.make(), out_end = events.make();
    if (in_end != nullptr && cudaEventRecord(in_end, cs.in) == cudaSuccess) cudaStreamWaitEvent(stream, in_end, 0);
    if (out_end != nullptr && cudaEventRecord(out_end, cs.out) == cudaSuccess) cudaStreamWaitEvent(stream, out_end, 0);
    return code;
  };

  const size_t row = static_cast<size_t>(d) * 2;  // bytes of one bf16 row
  const int g = Hq / Hkv;
  // Pieces: ranges [u0, u1) of the flattened (batch, key/value head) index
  // b * Hkv + h, contiguous in every tensor (a range may cross a batch
  // boundary: the kernel then sees its slices as the heads of one batch).
  // Sizes fall linearly from the first piece to the last (weights n, n-1,
  // ..., 1), so that the tail after the last input copy -- the last kernel
  // and the last output copy -- stays short.  A packed batch is one piece.
  struct Piece {
    long long u0, u1;
  };
  std::vector<Piece> list;
  const long long units = packed ? 1 : static_cast<long long>(B) * Hkv;
  {
    const long long n = units < pieces ? units : pieces;
    const long long wsum = n * (n + 1) / 2;
    long long u = 0;
    for (long long i = 0; i < n; ++i) {
      // Cumulative share of the first i + 1 weights, rounded; at least one unit per piece.
      const long long cum = n - 1 - i;  // weights left after this piece: 1 + ... + cum
      long long end = units - (units * (cum * (cum + 1) / 2) + wsum / 2) / wsum;
      if (end < u + 1) end = u + 1;
      if (end > units - (n - 1 - i)) end = units - (n - 1 - i);
      list.push_back(Piece{u, end});
      u = end;
    }
  }
  auto at = [](const void* base, size_t off) {
    return static_cast<void*>(static_cast<char*>(const_cast<void*>(base)) + off);
  };
  if (packed && !fa::copy(cu_seqlens_d, cu_seqlens_h, sizeof(int32_t) * (static_cast<size_t>(B) + 1),
                          cudaMemcpyHostToDevice, cs.in))
    return fail(FA_ERR_CUDA);
  for (const Piece& pc : list) {
    const int hkv = packed ? Hkv : static_cast<int>(pc.u1 - pc.u0), hq = hkv * g;
    // Dense: the piece's rows are contiguous in every tensor (batch-major, then head).
    const size_t q_rows0 = packed ? 0 : static_cast<size_t>(pc.u0) * g * Nq;
    const size_t kv_rows0 = packed ? 0 : static_cast<size_t>(pc.u0) * static_cast<size_t>(Nk);
    const size_t q_rows = static_cast<size_t>(hq) * Nq, kv_rows = static_cast<size_t>(hkv) * Nk;
    if (!fa::copy(at(q_d, q_rows0 * row), at(q_h, q_rows0 * row), q_rows * row, cudaMemcpyHostToDevice, cs.in) ||
        (Nk > 0 && (!fa::copy(at(k_d, kv_rows0 * row), at(k_h, kv_rows0 * row), kv_rows * row,
                              cudaMemcpyHostToDevice, cs.in) ||
                    !fa::copy(at(v_d, kv_rows0 * row), at(v_h, kv_rows0 * row), kv_rows * row,
                              cudaMemcpyHostToDevice, cs.in))))
      return fail(FA_ERR_CUDA);
    cudaEvent_t in_done = events.make();
    if (in_done == nullptr || cudaEventRecord(in_done, cs.in) != cudaSuccess ||
        cudaStreamWaitEvent(stream, in_done, 0) != cudaSuccess)
      return fail(FA_ERR_CUDA);
    st = fa_fwd(at(q_d, q_rows0 * row), Nk > 0 ? at(k_d, kv_rows0 * row) : nullptr,
                Nk > 0 ? at(v_d, kv_rows0 * row) : nullptr, at(o_d, q_rows0 * row),
                static_cast<float*>(at(lse_d, q_rows0 * sizeof(float))), packed ? B : 1, hq, hkv, Nq, Nk, d, scale,
                causal, packed ? cu_seqlens_d : nullptr, stream);
    if (st != FA_OK) return fail(st);
    cudaEvent_t k_done = events.make();
    if (k_done == nullptr || cudaEventRecord(k_done, stream) != cudaSuccess ||
        cudaStreamWaitEvent(cs.out, k_done, 0) != cudaSuccess)
      return fail(FA_ERR_CUDA);
    if (!fa::copy(at(o_h, q_rows0 * row), at(o_d, q_rows0 * row), q_rows * row, cudaMemcpyDeviceToHost, cs.out) ||
        !fa::copy(at(lse_h, q_rows0 * sizeof(float)), at(lse_d, q_rows0 * sizeof(float)), q_rows * sizeof(float),
                  cudaMemcpyDeviceToHost, cs.out))
      return fail(FA_ERR_CUDA);
  }
  // Later work on `stream` sees O and LSE in host memory.
  cudaEvent_t done = events.make();
  if (done == nullptr || cudaEventRecord(done, cs.out) != cudaSuccess ||
      cudaStreamWaitEvent(stream, done, 0) != cudaSuccess)
    return fail(FA_ERR_CUDA);
  return FA_OK;
}
