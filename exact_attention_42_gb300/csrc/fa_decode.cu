// Split-KV attention for few query rows per key/value head (decode).
//
// With a handful of query tokens against a long context the work is bound
// by reading K and V from HBM: each new token has to read the K/V of every
// earlier token (KV-cache overview canvas, element text-0023).  So this
// path streams K/V once at full bandwidth instead of padding a 128-row
// tensor-core tile.  It computes exactly what fa_fwd computes (same masks,
// outputs and statistics) for dense inputs.
//
// Decomposition: one thread-block cluster per (batch, key/value head); the S
// CTAs of a cluster split the key range.  Each CTA handles every query row
// of its head group, R = (Hq / Hkv) * Nq <= 16 rows: query head h = kvh*g +
// r / Nq, query token r % Nq.  A producer warp streams the CTA's keys in
// 128-key K/V tiles through a TMA ring (full / empty mbarriers); eight compute
// warps each own 16 keys of every tile and keep their own online-softmax
// state (reference max m, sum l, output accumulator; interview canvas,
// elements formula-text and qa2-a) for all R rows, so no CTA-wide barrier is
// needed per tile.  At the end the warp states, then the CTA states of the
// cluster (through distributed shared memory), are merged with
// m* = max m_s, l* = sum l_s 2^(m_s - m*), O* = sum O_s 2^(m_s - m*) / l*.
// No global scratch memory is used.
//
// Both products are small dense contractions on warp-level bf16 mma.sync
// (m16n8k16, fp32 accumulation) with the query rows as the M = 16 side:
// S = Q K^T takes Q fragments that stay in registers for the whole kernel and
// K fragments read by ldmatrix from the swizzled TMA tile; the fp32 score
// fragments of a warp's 16 keys, exponentiated and rounded to bf16, are
// exactly the A operand of O += P V, whose V fragments come from
// ldmatrix.trans.  Scores are in base 2 (scaled by scale * log2(e)); the
// reference max moves only when a tile's max exceeds it by more than 8, so
// most tiles skip the rescale of O.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <cmath>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace dec {

constexpr int COMPUTE_WARPS = 8;
constexpr int THREADS = 32 * (COMPUTE_WARPS + 1);  // + one TMA producer warp
constexpr int KEYS_PER_WARP = 16;
constexpr int BLOCK_N = KEYS_PER_WARP * COMPUTE_WARPS;  // 128 keys per tile
constexpr int MAX_R = 16;                                // query rows per key/value head (the MMA's M)
constexpr int MAX_SPLITS = 8;                            // portable cluster size
constexpr float RESCALE_TAU = 8.f;                       // reference-max slack (log2 units)

template <int D>
struct Cfg {
  static constexpr int STAGES = D == 128 ? 3 : 6;
  static constexpr int CHUNKS = D / 64;                 // 128-byte column blocks
  static constexpr int CHUNK_BYTES = BLOCK_N * 128;     // 16 KB
  static constexpr int TILE_BYTES = BLOCK_N * D * 2;    // one K or V tile
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int SMEM_RING = STAGES * STAGE_BYTES;
  static constexpr int SMEM_O = MAX_R * D * 4;                  // CTA partial O for the merge
  static constexpr int SMEM_WSTATS = 2 * COMPUTE_WARPS * MAX_R * 4;  // per-warp m, l
  static constexpr int SMEM_STATS = 2 * MAX_R * 4;              // CTA m, l
  static constexpr int SMEM_BYTES = 1024 + SMEM_RING + SMEM_O + SMEM_WSTATS + SMEM_STATS + 2 * STAGES * 8 + 16;
  static_assert(COMPUTE_WARPS * MAX_R * D * 4 <= SMEM_RING, "the warp merge is staged in the ring");
};

struct Params {
  const __nv_bfloat16* q;
  __nv_bfloat16* o;
  float* lse;
  int B, Hq, Hkv, Nq, Nk, group, R;
  float scale_log2;
  int causal;
  int keys_per_split;  // multiple of BLOCK_N
  unsigned long long wait_limit_ns;
  int fault_inject;    // test hook: 1 = every producer withholds its first tile
};

__device__ int g_decode_status;

// Byte offset of element (row, col) in a [chunk][64 rows][64 cols] bf16 tile
// written by TMA with the 128-byte swizzle (16-byte chunk index XOR row % 8).
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return static_cast<uint32_t>((col >> 6) * (BLOCK_N * 128) + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
                               ((col & 7) << 1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D += A B for a 16x8x16 bf16 tile, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, const Params p) {
  using C = Cfg<D>;
  constexpr int STAGES = C::STAGES;
  constexpr int KSTEPS = D / 16;  // k-steps of S = Q K^T
  constexpr int NTILES = D / 8;   // 8-dim output tiles of O += P V
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sRing = smem;
  float* sO = reinterpret_cast<float*>(smem + C::SMEM_RING);
  float* sMw = sO + MAX_R * D;               // [COMPUTE_WARPS][MAX_R]
  float* sLw = sMw + COMPUTE_WARPS * MAX_R;  // [COMPUTE_WARPS][MAX_R]
  float* sM = sLw + COMPUTE_WARPS * MAX_R;
  float* sL = sM + MAX_R;
  uint64_t* full = reinterpret_cast<uint64_t*>(sL + MAX_R);
  uint64_t* empty = full + STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + STAGES);

  const int tid = threadIdx.x;
  const int warp = tid / 32, lane = tid % 32;
  const int split = static_cast<int>(cluster_ctarank());
  const int nsplit = static_cast<int>(gridDim.x);
  const int bh = blockIdx.y;
  const int b = bh / p.Hkv, kvh = bh % p.Hkv;
  const int k_begin = split * p.keys_per_split;
  const int k_end = min(p.Nk, k_begin + p.keys_per_split);
  const int ntiles = k_end > k_begin ? (k_end - k_begin + BLOCK_N - 1) / BLOCK_N : 0;
  const int R = p.R;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), COMPUTE_WARPS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Set-up above overlaps the previous kernel's tail; global memory only after it.
  grid_dependency_wait();
  if (tid == 0) grid_launch_dependents();

  // Online-softmax state of a compute warp for fragment rows g and g + 8
  // (g = lane / 4): reference max m, partial sum l, output fragments o.
  const int g = lane / 4, q4 = lane % 4;
  const int r0 = g, r1 = g + 8;
  float o[NTILES][4];
#pragma unroll
  for (int n = 0; n < NTILES; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  if (warp == COMPUTE_WARPS) {
    // ---- TMA producer: tile t goes to stage t % STAGES once its previous
    // occupant has been released by every compute warp.
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int issued = 0;
      int withheld = -1;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % STAGES;
        if (t >= STAGES &&
            !mbar_wait(smem_u32(&empty[s]), ((t / STAGES) - 1) & 1u, abort_flag, p.wait_limit_ns)) {
          if (!*abort_flag) {
            *abort_flag = 1;
            atomicOr(&g_decode_status, 1);
          }
          break;
        }
        if (p.fault_inject && t == 0) {  // test hook: this tile never arrives
          withheld = t;
          issued = t + 1;
          continue;
        }
        const uint32_t bar = smem_u32(&full[s]);
        mbar_arrive_expect_tx(bar, C::STAGE_BYTES);
        const uint32_t dst = smem_u32(sRing + s * C::STAGE_BYTES);
        const int row = k_begin + t * BLOCK_N;
#pragma unroll
        for (int c = 0; c < C::CHUNKS; ++c) {
          tma_load_3d(dst + c * C::CHUNK_BYTES, &tm_k, bar, c * 64, row, bh);
          tma_load_3d(dst + C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_v, bar, c * 64, row, bh);
        }
        issued = t + 1;
      }
      // After an abort, wait (bounded, ignoring the flag) for the copies still
      // in flight before the shared memory is released.
      if (*abort_flag) {
        __shared__ int never;
        never = 0;
        for (int t = max(0, issued - STAGES); t < issued; ++t)
          if (t != withheld) mbar_wait(smem_u32(&full[t % STAGES]), (t / STAGES) & 1u, &never, p.wait_limit_ns);
      }
    }
    __syncwarp();
  } else {
    // ---- compute warp: keys [16 warp, +16) of every tile, all query rows.
    uint32_t qa[KSTEPS][4];  // A operand of S = Q K^T (rows >= R are zero)
    {
      const uint32_t* row_ptr[2];
      bool valid[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int r = h2 ? r1 : r0;
        valid[h2] = r < R;
        const int h = kvh * p.group + (valid[h2] ? r / p.Nq : 0), i = valid[h2] ? r % p.Nq : 0;
        row_ptr[h2] =
            reinterpret_cast<const uint32_t*>(p.q + ((static_cast<long long>(b) * p.Hq + h) * p.Nq + i) * D);
      }
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        const int c = 8 * ks + q4;  // 32-bit word of head dims 16 ks + 2 q4, +1
        qa[ks][0] = valid[0] ? __ldg(row_ptr[0] + c) : 0u;
        qa[ks][1] = valid[1] ? __ldg(row_ptr[1] + c) : 0u;
        qa[ks][2] = valid[0] ? __ldg(row_ptr[0] + c + 4) : 0u;
        qa[ks][3] = valid[1] ? __ldg(row_ptr[1] + c + 4) : 0u;
      }
    }
    // Last visible key of each fragment row, and the first key any row masks.
    const int shift = p.Nk - p.Nq;
    const int lim0 = p.causal ? min(k_end - 1, r0 % p.Nq + shift) : k_end - 1;
    const int lim1 = p.causal ? min(k_end - 1, r1 % p.Nq + shift) : k_end - 1;
    const int mask_from = p.causal ? min(k_end - 1, shift) : k_end - 1;
    const int kw = KEYS_PER_WARP * warp;  // first key of this warp in a tile

    for (int t = 0; t < ntiles; ++t) {
      const int s = t % STAGES;
      const bool got = mbar_wait(smem_u32(&full[s]), (t / STAGES) & 1u, abort_flag, p.wait_limit_ns);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0 && !*abort_flag) {
          *abort_flag = 1;
          atomicOr(&g_decode_status, 1);
        }
        break;
      }
      const uint32_t sK = smem_u32(sRing + s * C::STAGE_BYTES);
      const uint32_t sV = sK + C::TILE_BYTES;

      // S = Q K^T over this warp's 16 keys as two n-tiles of 8 keys;
      // sc[j][e] is row (e < 2 ? r0 : r1), key kw + 8 j + 2 q4 + e % 2.
      float sc[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
        for (int k2 = 0; k2 < KSTEPS / 2; ++k2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(sK + swz(kw + 8 * j + (lane % 8), 32 * k2 + 8 * (lane / 8)), b0, b1, b2, b3);
          mma_bf16_16816(sc[j], qa[2 * k2][0], qa[2 * k2][1], qa[2 * k2][2], qa[2 * k2][3], b0, b1);
          mma_bf16_16816(sc[j], qa[2 * k2 + 1][0], qa[2 * k2 + 1][1], qa[2 * k2 + 1][2], qa[2 * k2 + 1][3], b2,
                         b3);
        }
      }
      const int key0 = k_begin + t * BLOCK_N;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[j][e] *= p.scale_log2;
      if (key0 + BLOCK_N - 1 > mask_from) {
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int kg = key0 + kw + 8 * j + 2 * q4 + (e % 2);
            if (kg > (e < 2 ? lim0 : lim1)) sc[j][e] = -INFINITY;
          }
      }
      float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      // A row's reference max moves only when this tile exceeds it by more
      // than RESCALE_TAU; its sum and output are rescaled then.
      const bool up0 = mx0 > m0 + RESCALE_TAU, up1 = mx1 > m1 + RESCALE_TAU;
      if (__any_sync(0xffffffffu, up0 || up1)) {
        float a0 = 1.f, a1 = 1.f;
        if (up0) {
          a0 = (m0 == -INFINITY) ? 0.f : ex2_approx(m0 - mx0);
          m0 = mx0;
        }
        if (up1) {
          a1 = (m1 == -INFINITY) ? 0.f : ex2_approx(m1 - mx1);
          m1 = mx1;
        }
        l0 *= a0;
        l1 *= a1;
#pragma unroll
        for (int n = 0; n < NTILES; ++n) {
          o[n][0] *= a0;
          o[n][1] *= a0;
          o[n][2] *= a1;
          o[n][3] *= a1;
        }
      }
      const float base0 = (m0 == -INFINITY) ? 0.f : m0, base1 = (m1 == -INFINITY) ? 0.f : m1;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        sc[j][0] = ex2_approx(sc[j][0] - base0);
        sc[j][1] = ex2_approx(sc[j][1] - base0);
        sc[j][2] = ex2_approx(sc[j][2] - base1);
        sc[j][3] = ex2_approx(sc[j][3] - base1);
        l0 += sc[j][0] + sc[j][1];
        l1 += sc[j][2] + sc[j][3];
      }
      // The two score n-tiles, rounded to bf16, are the A operand of P V.
      const uint32_t pa0 = pack_bf16x2(sc[0][0], sc[0][1]), pa1 = pack_bf16x2(sc[0][2], sc[0][3]);
      const uint32_t pa2 = pack_bf16x2(sc[1][0], sc[1][1]), pa3 = pack_bf16x2(sc[1][2], sc[1][3]);
#pragma unroll
      for (int n2 = 0; n2 < NTILES / 2; ++n2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_trans(sV + swz(kw + (lane % 8) + 8 * ((lane / 8) % 2), 16 * n2 + 8 * (lane / 16)), b0, b1, b2,
                      b3);
        mma_bf16_16816(o[2 * n2], pa0, pa1, pa2, pa3, b0, b1);
        mma_bf16_16816(o[2 * n2 + 1], pa0, pa1, pa2, pa3, b2, b3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if (q4 == 0) {
      sMw[warp * MAX_R + r0] = m0;
      sLw[warp * MAX_R + r0] = l0;
      sMw[warp * MAX_R + r1] = m1;
      sLw[warp * MAX_R + r1] = l1;
    }
  }
  __syncthreads();
  // ---- merge the compute warps into this CTA's state (sM, sL, sO).  The
  // ring is idle now; each warp stages its rescaled output there and the sum
  // over warps is taken in a fixed order, so results do not vary run to run.
  float* sOw = reinterpret_cast<float*>(sRing);  // [COMPUTE_WARPS][MAX_R][D]
  if (warp < COMPUTE_WARPS) {
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int r = h2 ? r1 : r0;
      if (r >= R) continue;
      float mc = -INFINITY;
#pragma unroll
      for (int w = 0; w < COMPUTE_WARPS; ++w) mc = fmaxf(mc, sMw[w * MAX_R + r]);
      const float mw = h2 ? m1 : m0;
      const float f = (mw == -INFINITY) ? 0.f : ex2_approx(mw - mc);
      float* dst = sOw + (warp * MAX_R + r) * D + 2 * q4;
#pragma unroll
      for (int n = 0; n < NTILES; ++n)
        *reinterpret_cast<float2*>(dst + 8 * n) = make_float2(o[n][2 * h2] * f, o[n][2 * h2 + 1] * f);
      if (warp == 0 && q4 == 0) {
        float lc = 0.f;
#pragma unroll
        for (int w = 0; w < COMPUTE_WARPS; ++w) {
          const float ms = sMw[w * MAX_R + r];
          if (ms != -INFINITY) lc += sLw[w * MAX_R + r] * ex2_approx(ms - mc);
        }
        sM[r] = mc;
        sL[r] = lc;
      }
    }
  }
  __syncthreads();
  for (int idx = tid; idx < R * D; idx += THREADS) {
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < COMPUTE_WARPS; ++w) acc += sOw[w * MAX_R * D + idx];
    sO[idx] = acc;
  }
  __syncthreads();
  // ---- merge the CTAs of the cluster through distributed shared memory
  cluster_sync_all();
  if (split == 0 && !*abort_flag) {
    const uint32_t base_m = smem_u32(sM), base_l = smem_u32(sL), base_o = smem_u32(sO);
    for (int idx = tid; idx < R * D; idx += THREADS) {
      const int r = idx / D, c = idx % D;
      float m_star = -INFINITY;
      for (int s = 0; s < nsplit; ++s) m_star = fmaxf(m_star, ld_cluster_f32(cluster_addr(base_m + 4 * r, s)));
      float l_star = 0.f, o_star = 0.f;
      if (m_star != -INFINITY) {
        for (int s = 0; s < nsplit; ++s) {
          const float ms = ld_cluster_f32(cluster_addr(base_m + 4 * r, s));
          if (ms == -INFINITY) continue;
          const float w = ex2_approx(ms - m_star);
          l_star += w * ld_cluster_f32(cluster_addr(base_l + 4 * r, s));
          o_star += w * ld_cluster_f32(cluster_addr(base_o + 4 * idx, s));
        }
      }
      const int h = kvh * p.group + r / p.Nq, i = r % p.Nq;
      const long long row = (static_cast<long long>(b) * p.Hq + h) * p.Nq + i;
      p.o[row * D + c] = __float2bfloat16(l_star > 0.f ? o_star / l_star : 0.f);
      if (c == 0) p.lse[row] = l_star > 0.f ? (m_star + __log2f(l_star)) * 0.69314718055994531f : -INFINITY;
    }
  }
  cluster_sync_all();  // the other splits keep their shared memory until the merge has read it
}

}  // namespace dec

// --------------------------------------------------------------------------
// Host side
// --------------------------------------------------------------------------

static bool encode_decode_map(CUtensorMap* map, const void* base, int d, long long rows, long long heads) {
  return encode_bf16_rows_map(map, base, d, rows, heads, dec::BLOCK_N);
}

bool decode_supported(int B, int Hq, int Hkv, int Nq, int Nk, int d, const int32_t* cu_seqlens) {
  (void)B;
  (void)d;
  return cu_seqlens == nullptr && Nk > 0 && Nq > 0 && (Hq / Hkv) * Nq <= dec::MAX_R;
}

template <int D>
static fa_status launch_decode_t(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                 int Hkv, int Nq, int Nk, float scale, int causal, cudaStream_t stream, int sms,
                                 unsigned long long wait_limit_ns, int fault_mode) {
  {
    static std::mutex mu;
    static bool attr_set[kMaxDevicesDecode] = {};
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    if (dev >= 0 && dev < kMaxDevicesDecode && !attr_set[dev]) {
      if (cudaFuncSetAttribute(dec::decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               dec::Cfg<D>::SMEM_BYTES) != cudaSuccess)
        return FA_ERR_CUDA;
      attr_set[dev] = true;
    }
  }
  alignas(64) CUtensorMap tk, tv;
  if (!encode_decode_map(&tk, k, D, Nk, static_cast<long long>(B) * Hkv) ||
      !encode_decode_map(&tv, v, D, Nk, static_cast<long long>(B) * Hkv))
    return FA_ERR_CUDA;
  const long long groups = static_cast<long long>(B) * Hkv;
  if (groups > 65535) return FA_ERR_SHAPE;
  // One CTA per SM: enough splits for the clusters to fill the SMs once,
  // each split at least two tiles long.
  long long S = groups >= sms ? 1 : sms / groups;
  S = S < 1 ? 1 : (S > dec::MAX_SPLITS ? dec::MAX_SPLITS : S);
  const long long max_by_len = (Nk + dec::BLOCK_N - 1) / dec::BLOCK_N / 2;
  if (S > max_by_len) S = max_by_len < 1 ? 1 : max_by_len;
  long long kps = (Nk + S - 1) / S;
  kps = (kps + dec::BLOCK_N - 1) / dec::BLOCK_N * dec::BLOCK_N;
  S = (Nk + kps - 1) / kps;

  dec::Params prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Nq = Nq;
  prm.Nk = Nk;
  prm.group = Hq / Hkv;
  prm.R = prm.group * Nq;
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  prm.causal = causal ? 1 : 0;
  prm.keys_per_split = static_cast<int>(kps);
  prm.wait_limit_ns = wait_limit_ns;
  prm.fault_inject = fault_mode == kFaultDecode ? 1 : 0;

  // One cluster of S CTAs per (batch, key/value head); clusters of one CTA are
  // still launched as clusters so that the split merge code is the same.
  PdlLaunch L(dim3(static_cast<unsigned>(S), static_cast<unsigned>(groups), 1), dec::THREADS,
              dec::Cfg<D>::SMEM_BYTES, stream, static_cast<unsigned>(S));
  L.cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&L.cfg, dec::decode_kernel<D>, tk, tv, prm) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

fa_status launch_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int Nq, int Nk, int d, float scale, int causal, cudaStream_t stream, int sms,
                        unsigned long long wait_limit_ns, int fault_mode) {
  if (d == 128)
    return launch_decode_t<128>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, stream, sms, wait_limit_ns,
                                fault_mode);
  return launch_decode_t<64>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, stream, sms, wait_limit_ns,
                             fault_mode);
}

int decode_status_and_clear() {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, dec::g_decode_status, sizeof(int)) != cudaSuccess) return -1;
  const int zero = 0;
  if (cudaMemcpyToSymbol(dec::g_decode_status, &zero, sizeof(int)) != cudaSuccess) return -1;
  return v;
}

int decode_smem_bytes(int d) {
  if (d == 64) return dec::Cfg<64>::SMEM_BYTES;
  if (d == 128) return dec::Cfg<128>::SMEM_BYTES;
  return 0;
}

}  // namespace fa
