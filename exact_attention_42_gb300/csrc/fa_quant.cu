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
// Four launches: zero the slice maxima (accumulated in the descale buffer
// itself), slice maxima, codes, descales.  No other memory is used.

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cmath>
#include <cstdint>

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
cudaError_t launch(const Args& a, int slices, bool transpose, cudaStream_t stream) {
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

}  // namespace quant

fa_status launch_fp8_quantize(const void* x, void* x8, float* descale, int B, int H, int N, int d, int transpose,
                              const int8_t* signs, cudaStream_t stream) {
  quant::Args a;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.x8 = static_cast<uint8_t*>(x8);
  a.descale = descale;
  a.signs = signs;
  a.N = N;
  a.tiles = (N + quant::ROWS_PER_BLOCK - 1) / quant::ROWS_PER_BLOCK;
  const int slices = B * H;
  const cudaError_t e = d == 128 ? quant::launch<128>(a, slices, transpose != 0, stream)
                                 : quant::launch<64>(a, slices, transpose != 0, stream);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace fa
