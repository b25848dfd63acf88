// Quantization of a bf16 tensor to e4m3 codes for the 8-bit forward, with
// one descale per (batch, head) slice and, optionally, the incoherent
// processing rotation first.
//
// The FA3 canvas ("FlashAttention v3 Hopper asynchrony: TMA + WGMMA +
// ping-pong", element pseudo-code) and the interview canvas
// ("FlashAttention面试讲解", element script-body) name block scaling of
// Q/K/V and incoherent processing as the two measures that keep the 8-bit
// path accurate.  Here a block is one (batch, head) slice of the tensor.  The
// rotation multiplies every row by M = diag(signs) H_d / sqrt(d), where H_d is
// the Sylvester-Hadamard matrix (entries +-1, H H^T = d I) and signs is a
// caller-drawn +-1 vector.  M is orthogonal, so rotating Q and K with the same
// signs leaves Q K^T unchanged while spreading a large channel over all d.
//
// Arithmetic, chosen so that a float32 CPU model reproduces every code:
//   y   = (x * signs) H_d, by the radix-2 Walsh-Hadamard butterflies with
//         strides 1, 2, 4, ... d/2 (lower <- a + b, upper <- a - b), float32;
//   a   = max |y| over the slice;
//   inv = 448 / a (float32, correctly rounded; 0 when a = 0);
//   code = e4m3(y * inv), round to nearest even, saturating at +-448;
//   descale = a / (448 sqrt(d)) with rotation, a / 448 without (float64, then
//         float32), so that code * descale approximates x M (or x).
// A slice that fits in the shared memory of one thread-block cluster is
// quantized in one launch (quant_fused_kernel, below).  Larger slices take
// four launches: zero the slice maxima (accumulated in the descale buffer
// itself), slice maxima, codes, descales.  No other memory is used.

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace quant {

constexpr int ROWS_PER_BLOCK = 64;
constexpr int THREADS = 128;  // four warps of 16 rows each
constexpr int ROWS_PER_WARP = ROWS_PER_BLOCK / (THREADS / 32);
// Rows a warp loads before using any of them: one 256-byte row in flight per
// warp left the kernels at about a third of the HBM bandwidth.
constexpr int BATCH = 8;
static_assert(ROWS_PER_WARP % BATCH == 0, "a warp's rows come in whole batches");

// Lane l holds columns [l * E, l * E + E) of a row, E = D / 32.
template <int D>
__device__ __forceinline__ void load_row(const __nv_bfloat16* row, int lane, float (&v)[D / 32]) {
  if constexpr (D == 128) {
    const uint2 raw = *reinterpret_cast<const uint2*>(row + lane * 4);
    v[0] = __uint_as_float(raw.x << 16);
    v[1] = __uint_as_float(raw.x & 0xffff0000u);
    v[2] = __uint_as_float(raw.y << 16);
    v[3] = __uint_as_float(raw.y & 0xffff0000u);
  } else {
    const uint32_t raw = *reinterpret_cast<const uint32_t*>(row + lane * 2);
    v[0] = __uint_as_float(raw << 16);
    v[1] = __uint_as_float(raw & 0xffff0000u);
  }
}

// (x * signs) H_d for the row held by the warp.
template <int D>
__device__ __forceinline__ void rotate_row(float (&v)[D / 32], const float (&sg)[D / 32], int lane) {
  constexpr int E = D / 32;
#pragma unroll
  for (int i = 0; i < E; ++i) v[i] = v[i] * sg[i];  // exact: sg is +-1
#pragma unroll
  for (int h = 1; h < E; h <<= 1) {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = __fadd_rn(a, b);
        v[i + h] = __fsub_rn(a, b);
      }
    }
  }
#pragma unroll
  for (int h = E; h < D; h <<= 1) {
    const int lm = h / E;  // partner lane distance
    const bool upper = (lane & lm) != 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float other = __shfl_xor_sync(0xffffffffu, v[i], lm);
      v[i] = upper ? __fsub_rn(other, v[i]) : __fadd_rn(v[i], other);
    }
  }
}

template <int D>
__device__ __forceinline__ void load_signs(const int8_t* signs, int lane, float (&sg)[D / 32]) {
#pragma unroll
  for (int i = 0; i < D / 32; ++i) sg[i] = signs[lane * (D / 32) + i] < 0 ? -1.f : 1.f;
}

// Two floats to two e4m3 codes (first argument in the low byte).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

struct Args {
  const __nv_bfloat16* x;  // [slices, N, D]
  uint8_t* x8;             // [slices, N, D] or [slices, D, N]
  float* descale;          // [slices]; holds the slice maxima (as bits) between the first two launches
  const int8_t* signs;     // [D] or nullptr
  int N;
  int tiles;               // blocks per slice
  int fault_inject;        // test hook (one-launch path): 1 = the first bulk copy of every CTA is withheld
};

// Zeroes the slice-maximum accumulators (the descale buffer).
__global__ void zero_kernel(float* descale, int slices) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < slices) descale[i] = 0.f;
}

template <int D>
__global__ void __launch_bounds__(THREADS) amax_kernel(const Args a) {
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  const int slice = blockIdx.x / a.tiles;
  const int r0 = (blockIdx.x % a.tiles) * ROWS_PER_BLOCK + (threadIdx.x / 32) * ROWS_PER_WARP;
  const int lane = threadIdx.x % 32;
  float sg[D / 32];
  if (a.signs != nullptr) load_signs<D>(a.signs, lane, sg);
  float m = 0.f;
  for (int rb = r0; rb < min(r0 + ROWS_PER_WARP, a.N); rb += BATCH) {
    float v[BATCH][D / 32];
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      if (rb + b < a.N) {
        load_row<D>(a.x + (static_cast<long long>(slice) * a.N + rb + b) * D, lane, v[b]);
      } else {
#pragma unroll
        for (int i = 0; i < D / 32; ++i) v[b][i] = 0.f;
      }
    }
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      if (a.signs != nullptr) rotate_row<D>(v[b], sg, lane);
#pragma unroll
      for (int i = 0; i < D / 32; ++i) m = fmaxf(m, fabsf(v[b][i]));
    }
  }
  // Non-negative floats order like their bit patterns.
  const uint32_t bits = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
  if (lane == 0 && bits != 0u) atomicMax(reinterpret_cast<unsigned int*>(a.descale) + slice, bits);
}

template <int D, bool TRANSPOSE>
__global__ void __launch_bounds__(THREADS) quant_kernel(const Args a) {
  constexpr int E = D / 32;
  constexpr int PITCH = D + 4;  // bytes per staged row; the 4-byte pad spreads a column over the banks
  __shared__ uint8_t tile[TRANSPOSE ? ROWS_PER_BLOCK * PITCH : 1];
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  const int slice = blockIdx.x / a.tiles;
  const int tile_r0 = (blockIdx.x % a.tiles) * ROWS_PER_BLOCK;
  const int r0 = tile_r0 + (threadIdx.x / 32) * ROWS_PER_WARP;
  const int lane = threadIdx.x % 32;
  float sg[E];
  if (a.signs != nullptr) load_signs<D>(a.signs, lane, sg);
  const float amax = __uint_as_float(__ldg(reinterpret_cast<const unsigned int*>(a.descale) + slice));
  const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
  for (int rb = r0; rb < min(r0 + ROWS_PER_WARP, a.N); rb += BATCH) {
    float v[BATCH][E];
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      if (rb + b < a.N) {
        load_row<D>(a.x + (static_cast<long long>(slice) * a.N + rb + b) * D, lane, v[b]);
      } else {
#pragma unroll
        for (int i = 0; i < E; ++i) v[b][i] = 0.f;
      }
    }
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      const int r = rb + b;
      if (a.signs != nullptr) rotate_row<D>(v[b], sg, lane);  // every lane takes part in the shuffles
      if (r >= a.N) continue;
      uint32_t packed = 0u;  // E codes, column lane * E first
#pragma unroll
      for (int i = 0; i < E; i += 2)
        packed |= e4m3x2(__fmul_rn(v[b][i], inv), __fmul_rn(v[b][i + 1], inv)) << (8 * i);
      if constexpr (TRANSPOSE) {
        uint8_t* dst = tile + (r - tile_r0) * PITCH + lane * E;
#pragma unroll
        for (int i = 0; i < E; ++i) dst[i] = static_cast<uint8_t>(packed >> (8 * i));
      } else {
        uint8_t* dst = a.x8 + (static_cast<long long>(slice) * a.N + r) * D + lane * E;
        if constexpr (E == 4)
          *reinterpret_cast<uint32_t*>(dst) = packed;
        else
          *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(packed);
      }
    }
  }
  if constexpr (TRANSPOSE) {
    __syncthreads();
    // Row c of the slice's transpose takes keys [tile_r0, tile_r0 + nrows) of
    // column c, 16 keys per thread and store (N and nrows are multiples of 16).
    const int nrows = min(ROWS_PER_BLOCK, a.N - tile_r0);
    const int per_col = nrows / 16;
    for (int q = threadIdx.x; q < D * per_col; q += THREADS) {
      const int c = q / per_col, part = q % per_col;
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t word = 0u;
#pragma unroll
        for (int b = 0; b < 4; ++b) word |= static_cast<uint32_t>(tile[(part * 16 + 4 * j + b) * PITCH + c]) << (8 * b);
        w[j] = word;
      }
      uint8_t* dst = a.x8 + (static_cast<long long>(slice) * D + c) * a.N + tile_r0 + part * 16;
      *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

__global__ void descale_kernel(float* descale, int slices, double divisor) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < slices) descale[i] = static_cast<float>(static_cast<double>(descale[i]) / divisor);
}

// Four launches, each with programmatic stream serialization (PdlLaunch):
// zero the accumulators, slice maxima, codes, descales.
template <int D>
cudaError_t launch_passes(const Args& a, int slices, bool transpose, cudaStream_t stream) {
  const long long blocks = static_cast<long long>(slices) * a.tiles;
  const unsigned small = static_cast<unsigned>((slices + 255) / 256);
  {
    PdlLaunch L(dim3(small), 256, 0, stream);
    const cudaError_t e = cudaLaunchKernelEx(&L.cfg, zero_kernel, a.descale, slices);
    if (e != cudaSuccess) return e;
  }
  if (blocks == 0) return cudaSuccess;  // no rows: every descale is 0
  {
    PdlLaunch L(dim3(static_cast<unsigned>(blocks)), THREADS, 0, stream);
    const cudaError_t e = cudaLaunchKernelEx(&L.cfg, amax_kernel<D>, a);
    if (e != cudaSuccess) return e;
  }
  {
    PdlLaunch L(dim3(static_cast<unsigned>(blocks)), THREADS, 0, stream);
    const cudaError_t e = transpose ? cudaLaunchKernelEx(&L.cfg, quant_kernel<D, true>, a)
                                    : cudaLaunchKernelEx(&L.cfg, quant_kernel<D, false>, a);
    if (e != cudaSuccess) return e;
  }
  const double divisor = 448.0 * (a.signs != nullptr ? std::sqrt(static_cast<double>(D)) : 1.0);
  PdlLaunch L(dim3(small), 256, 0, stream);
  return cudaLaunchKernelEx(&L.cfg, descale_kernel, a.descale, slices, divisor);
}


// ---------------------------------------------------------------------------
// One-launch path: one thread-block cluster of `ncta` CTAs per slice.  CTA
// rank r copies rows [r R, r R + R) of its slice into shared memory with bulk
// copies (64-row pieces, one mbarrier each), takes their maximum, and the
// cluster combines the CTA maxima through distributed shared memory; then
// every CTA writes the codes of its rows from shared memory.  x is read from
// HBM once, and no atomics, accumulator or memset are needed.  The arithmetic
// is the same as the three-kernel path's (same butterflies, division and
// conversion), so codes and descales are identical.
// ---------------------------------------------------------------------------
constexpr int FTHREADS = 256;  // 8 warps
constexpr int FWARPS = FTHREADS / 32;
constexpr int FCHUNK = 64;     // rows per bulk copy (and per transposed staging tile)
constexpr int FMAX_CTAS = 16;  // cluster size limit (16 is above the portable 8)
constexpr int FMAX_SMEM_X = 64 * 1024;  // bytes of rows per CTA

__device__ int g_quant_status;  // set when a wait for the bulk copies ran out

template <int D>
constexpr int fused_smem(int rows_per_cta) {
  return rows_per_cta * D * 2 + FCHUNK * (D + 4) + 64 + (rows_per_cta / FCHUNK) * 8 + 16;
}

// Lane l's elements [l E, l E + E) of a bf16 row in shared memory.
template <int D>
__device__ __forceinline__ void load_row_smem(const __nv_bfloat16* row, int lane, float (&v)[D / 32]) {
  if constexpr (D == 128) {
    const uint2 raw = *reinterpret_cast<const uint2*>(row + lane * 4);
    v[0] = __uint_as_float(raw.x << 16);
    v[1] = __uint_as_float(raw.x & 0xffff0000u);
    v[2] = __uint_as_float(raw.y << 16);
    v[3] = __uint_as_float(raw.y & 0xffff0000u);
  } else {
    const uint32_t raw = *reinterpret_cast<const uint32_t*>(row + lane * 2);
    v[0] = __uint_as_float(raw << 16);
    v[1] = __uint_as_float(raw & 0xffff0000u);
  }
}

template <int D, bool TRANSPOSE>
__global__ void __launch_bounds__(FTHREADS) quant_fused_kernel(const Args a, int rows_per_cta, double divisor,
                                                               unsigned long long limit_ns) {
  constexpr int E = D / 32;
  constexpr int PITCH = D + 4;
  extern __shared__ __align__(128) uint8_t fsmem[];
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(fsmem);
  uint8_t* tile = fsmem + rows_per_cta * D * 2;
  float* wmax = reinterpret_cast<float*>(tile + FCHUNK * PITCH);  // [FWARPS], then the CTA maximum
  float* cmax = wmax + FWARPS;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(cmax + 1);
  uint64_t* bars = reinterpret_cast<uint64_t*>(fsmem + rows_per_cta * D * 2 + FCHUNK * PITCH + 64);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int ncta = static_cast<int>(cluster_nctarank());
  const int rank = static_cast<int>(cluster_ctarank());
  const int slice = static_cast<int>(blockIdx.x) / ncta;
  const int r0 = rank * rows_per_cta;
  const int nrows = max(0, min(a.N - r0, rows_per_cta));
  const int nchunks = (nrows + FCHUNK - 1) / FCHUNK;
  if (tid == 0) {
    for (int c = 0; c < nchunks; ++c) mbar_init(smem_u32(&bars[c]), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_wait();
  if (tid == 0) grid_launch_dependents();
  const __nv_bfloat16* src = a.x + (static_cast<long long>(slice) * a.N + r0) * D;
  if (tid == 0) {
    for (int c = 0; c < nchunks; ++c) {
      if (a.fault_inject && c == 0) continue;  // test hook: this copy never arrives
      const uint32_t bytes = static_cast<uint32_t>(min(FCHUNK, nrows - c * FCHUNK) * D * 2);
      mbar_arrive_expect_tx(smem_u32(&bars[c]), bytes);
      bulk_load(smem_u32(xs + c * FCHUNK * D), src + static_cast<long long>(c) * FCHUNK * D, bytes,
                smem_u32(&bars[c]));
    }
  }
  float sg[E];
  if (a.signs != nullptr) load_signs<D>(a.signs, lane, sg);
  // Maximum of |y| over this CTA's rows, chunk by chunk as the copies land.
  float m = 0.f;
  for (int c = 0; c < nchunks; ++c) {
    if (!mbar_wait(smem_u32(&bars[c]), 0, abort_flag, limit_ns)) {
      if (lane == 0 && !*abort_flag) {
        *abort_flag = 1;
        atomicOr(&g_quant_status, 1);
      }
      break;
    }
    // Warp w takes rows w, w + 8, ..., w + 56 of the chunk, all eight in flight.
    const int rend = min(FCHUNK, nrows - c * FCHUNK);
    float v[FCHUNK / FWARPS][E];
#pragma unroll
    for (int b = 0; b < FCHUNK / FWARPS; ++b) {
      const int r = warp + b * FWARPS;
      if (r < rend) {
        load_row_smem<D>(xs + (c * FCHUNK + r) * D, lane, v[b]);
      } else {
#pragma unroll
        for (int i = 0; i < E; ++i) v[b][i] = 0.f;
      }
    }
#pragma unroll
    for (int b = 0; b < FCHUNK / FWARPS; ++b) {
      if (a.signs != nullptr) rotate_row<D>(v[b], sg, lane);
#pragma unroll
      for (int i = 0; i < E; ++i) m = fmaxf(m, fabsf(v[b][i]));
    }
  }
  m = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(m)));  // non-negative floats order like their bits
  if (lane == 0) wmax[warp] = m;
  __syncthreads();
  if (tid == 0) {
    float cm = 0.f;
#pragma unroll
    for (int w = 0; w < FWARPS; ++w) cm = fmaxf(cm, wmax[w]);
    *cmax = cm;
  }
  cluster_sync_all();  // every CTA's maximum is in place
  float amax = 0.f;
  for (int r = 0; r < ncta; ++r) amax = fmaxf(amax, ld_cluster_f32(cluster_addr(smem_u32(cmax), r)));
  const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
  if (!*abort_flag) {
    for (int c = 0; c < nchunks; ++c) {
      const int rend = min(FCHUNK, nrows - c * FCHUNK);
      float v[FCHUNK / FWARPS][E];
#pragma unroll
      for (int b = 0; b < FCHUNK / FWARPS; ++b) {
        const int r = warp + b * FWARPS;
        if (r < rend) {
          load_row_smem<D>(xs + (c * FCHUNK + r) * D, lane, v[b]);
        } else {
#pragma unroll
          for (int i = 0; i < E; ++i) v[b][i] = 0.f;
        }
      }
#pragma unroll
      for (int b = 0; b < FCHUNK / FWARPS; ++b) {
        const int r = warp + b * FWARPS;
        if (a.signs != nullptr) rotate_row<D>(v[b], sg, lane);  // every lane takes part in the shuffles
        if (r >= rend) continue;
        uint32_t packed = 0u;  // E codes, column lane * E first
#pragma unroll
        for (int i = 0; i < E; i += 2)
          packed |= e4m3x2(__fmul_rn(v[b][i], inv), __fmul_rn(v[b][i + 1], inv)) << (8 * i);
        if constexpr (TRANSPOSE) {
          uint8_t* dst = tile + r * PITCH + lane * E;
#pragma unroll
          for (int i = 0; i < E; ++i) dst[i] = static_cast<uint8_t>(packed >> (8 * i));
        } else {
          uint8_t* dst = a.x8 + (static_cast<long long>(slice) * a.N + r0 + c * FCHUNK + r) * D + lane * E;
          if constexpr (E == 4)
            *reinterpret_cast<uint32_t*>(dst) = packed;
          else
            *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(packed);
        }
      }
      if constexpr (TRANSPOSE) {
        __syncthreads();
        // Column col of the slice's transpose takes keys [r0 + 64 c, + rend):
        // 16 keys per thread and store (N and rend are multiples of 16).
        const int per_col = rend / 16;
        for (int q = tid; q < D * per_col; q += FTHREADS) {
          const int col = q / per_col, part = q % per_col;
          uint32_t w[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t word = 0u;
#pragma unroll
            for (int b = 0; b < 4; ++b)
              word |= static_cast<uint32_t>(tile[(part * 16 + 4 * j + b) * PITCH + col]) << (8 * b);
            w[j] = word;
          }
          uint8_t* dst = a.x8 + (static_cast<long long>(slice) * D + col) * a.N + r0 + c * FCHUNK + part * 16;
          *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        __syncthreads();
      }
    }
  }
  if (rank == 0 && tid == 0) a.descale[slice] = static_cast<float>(static_cast<double>(amax) / divisor);
  if (*abort_flag && tid == 0) {
    // Copies still in flight land before the shared memory is released.
    __shared__ int never;
    never = 0;
    for (int c = 0; c < nchunks; ++c) mbar_wait(smem_u32(&bars[c]), 0, &never, limit_ns);
  }
  cluster_sync_all();  // no CTA leaves while another may still read its maximum
}

// Cluster size and rows per CTA of the one-launch path for a slice of N rows,
// or false when a slice does not fit in the shared memory of FMAX_CTAS CTAs.
template <int D>
static bool fused_shape(int N, int slices, int sms, int* ncta, int* rows) {
  const int max_rows = FMAX_SMEM_X / (D * 2);
  int c = 1;
  // Enough CTAs to fill the GPU twice over, and no more rows per CTA than fit.
  while (c < FMAX_CTAS && (static_cast<long long>(slices) * c < 2LL * sms || (N + c - 1) / c > max_rows)) c *= 2;
  int r = (N + c - 1) / c;
  r = (r + FCHUNK - 1) / FCHUNK * FCHUNK;
  if (r > max_rows || r <= 0) return false;
  *ncta = c;
  *rows = r;
  return true;
}

template <int D, bool TRANSPOSE>
static bool fused_ready(int ncta) {
  // Shared-memory limit once per device; cluster sizes above 8 need the non-portable opt-in.
  static std::mutex mu;
  static int state[kMaxDevicesDecode][2] = {};  // 0 unknown, 1 ready, 2 unavailable; [ncta > 8]
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesDecode) return false;
  std::lock_guard<std::mutex> lock(mu);
  int& st = state[dev][ncta > 8 ? 1 : 0];
  if (st == 0) {
    st = 2;
    const int smem = fused_smem<D>(FMAX_SMEM_X / (D * 2));
    if (cudaFuncSetAttribute(quant_fused_kernel<D, TRANSPOSE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
            cudaSuccess &&
        (ncta <= 8 ||
         cudaFuncSetAttribute(quant_fused_kernel<D, TRANSPOSE>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
             cudaSuccess)) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(ncta), 1, 1);
      cfg.blockDim = dim3(FTHREADS, 1, 1);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(ncta);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, quant_fused_kernel<D, TRANSPOSE>, &cfg) == cudaSuccess && n > 0) st = 1;
    }
    cudaGetLastError();  // a refused opt-in leaves the three-kernel path
  }
  return st == 1;
}

// Which path runs, from measurements on GB300 (CUDA events, 60 calls):
//   B4 H16 N1024 d64:  one launch 0.0105 ms against 0.0185 (all three kinds);
//   B2 H32 N4096 d128: one launch 0.030 ms against 0.033 unrotated, but
//   0.043 against 0.039 transposed and 0.078 against 0.058 rotated -- with
//   large slices the butterflies and the transpose staging want the higher
//   occupancy of the four-launch kernels.
template <int D>
cudaError_t launch(const Args& a, int slices, bool transpose, cudaStream_t stream, int sms,
                   unsigned long long limit_ns) {
  const double divisor = 448.0 * (a.signs != nullptr ? std::sqrt(static_cast<double>(D)) : 1.0);
  const bool one_launch = a.N <= 1024 || (a.signs == nullptr && !transpose);
  int ncta = 0, rows = 0;
  if (a.N > 0 && one_launch && fused_shape<D>(a.N, slices, sms, &ncta, &rows) &&
      (transpose ? fused_ready<D, true>(ncta) : fused_ready<D, false>(ncta))) {
    PdlLaunch L(dim3(static_cast<unsigned>(slices * ncta)), FTHREADS, fused_smem<D>(rows), stream,
                static_cast<unsigned>(ncta));
    L.cfg.numAttrs = 2;  // always a cluster launch (the kernel reads its cluster rank)
    return transpose ? cudaLaunchKernelEx(&L.cfg, quant_fused_kernel<D, true>, a, rows, divisor, limit_ns)
                     : cudaLaunchKernelEx(&L.cfg, quant_fused_kernel<D, false>, a, rows, divisor, limit_ns);
  }
  return launch_passes<D>(a, slices, transpose, stream);
}
}  // namespace quant

fa_status launch_fp8_quantize(const void* x, void* x8, float* descale, int B, int H, int N, int d, int transpose,
                              const int8_t* signs, cudaStream_t stream, const LaunchEnv& env) {
  quant::Args a;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.x8 = static_cast<uint8_t*>(x8);
  a.descale = descale;
  a.signs = signs;
  a.N = N;
  a.tiles = (N + quant::ROWS_PER_BLOCK - 1) / quant::ROWS_PER_BLOCK;
  a.fault_inject = env.fault_mode == kFaultQuant ? 1 : 0;
  const int slices = B * H;
  const cudaError_t e = d == 128 ? quant::launch<128>(a, slices, transpose != 0, stream, env.sms, env.wait_limit_ns)
                                 : quant::launch<64>(a, slices, transpose != 0, stream, env.sms, env.wait_limit_ns);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int quant_status_and_clear() {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, quant::g_quant_status, sizeof(int)) != cudaSuccess) return -1;
  const int zero = 0;
  if (cudaMemcpyToSymbol(quant::g_quant_status, &zero, sizeof(int)) != cudaSuccess) return -1;
  return v;
}

}  // namespace fa
