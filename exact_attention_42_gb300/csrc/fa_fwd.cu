// Exact attention forward for GB300 (sm_103a): tcgen05 tensor cores with
// S and O accumulators in Tensor Memory, TMA-fed K/V ring, warp-specialised
// load / MMA / softmax roles, and an online softmax with conditional rescale.
//
// Method ("FlashAttention面试讲解" interview canvas): K/V are moved tile by
// tile into on-chip memory and, for each tile, QK^T, the online softmax and
// the PV accumulation are done together so the N x N matrix never reaches HBM
// (element flash-text); the softmax keeps a running max m, a running sum l and
// the output accumulator O, and rescales old O and l by exp(m_old - m_new)
// when the max grows (elements formula-text, qa2-a).  The Blackwell notes of
// the same canvas (element v4-card-body) motivate the layout: accumulators in
// TMEM, a fully asynchronous MMA pipeline, and a conditional rescale.  The
// producer/consumer split and the idea of hiding one tile's softmax behind
// another tile's matrix products come from the Hopper pipeline canvas
// ("FlashAttention v3 Hopper asynchrony", elements pseudo-code and
// pipeline-note); here the two consumers are two 128-row Q tiles that share
// every K/V tile.
//
// CTA layout (384 threads, one CTA per SM, persistent over work units):
//   warps 0-3  softmax for Q tile 0 (thread r owns row r = TMEM lane r)
//   warps 4-7  softmax for Q tile 1
//   warp 8     K/V producer (one lane): K_j, V_j of every unit into the ring
//   warp 9     MMA issuer and TMEM owner: the whole warp runs the issue loop
//              and one elected lane issues, which keeps descriptors and loop
//              state warp-uniform (about 95 cycles per tcgen05.mma, against
//              about 130 when a lone lane runs the loop)
//   warp 10    idle
//   warp 11    Q loader (one lane): reloads Q tile t as soon as the last QK of
//              tile t in the previous unit has completed, so the K/V stream
//              never stalls at a unit boundary
// Products are issued in the order QK_0(0), QK_1(0), then per K/V tile j:
// PV_0(j), QK_0(j+1), PV_1(j), QK_1(j+1).  Tile 0's softmax therefore runs
// while the tensor pipe works on tile 1's products and the other way round.
// TMEM (512 columns x 128 lanes, fp32):
//   [0,128)   S_0   (P_0 as packed bf16 pairs overwrites columns [0,64))
//   [128,256) S_1   (P_1 likewise)
//   [256,384) O_0   [384,512) O_1   (d = 64 uses the first 64 of each)
// A work unit is 256 consecutive query rows (two tiles) of one head.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <cmath>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

constexpr int BLOCK_M = 128;      // query rows per tile (= TMEM lanes)
constexpr int BLOCK_N = 128;      // keys per K/V tile
constexpr int NQT = 2;            // query tiles per CTA
constexpr int NUM_THREADS = 384;  // three warpgroups
constexpr int WARP_PRODUCER = 8;
constexpr int WARP_MMA = 9;  // issues the products of both query tiles (warp 10 is idle)
constexpr int WARP_QLOAD = 11;
// Register split.  The kernel is launched at 168 registers per thread (the
// most 12 warps allow: three warps share each sub-partition's 16K registers).
// The two softmax warpgroups then grow to REG_SOFTMAX and the load/MMA
// warpgroup shrinks to REG_OTHER (per instantiation, see Cfg): bf16
// 8*216 + 4*72 = 2016 = 12*168 (the block's pool), 8-bit 8*224 + 4*56 = 2016;
// per sub-partition 2*216 + 72 = 504 and 2*224 + 56 = 504 <= 512.  The 8-bit
// softmax needs more registers (ptxas: 44 bytes of spills at 216, 28 at
// 224), and 224/56 measured 0.6-0.7% faster there; bf16 compiles without
// spills at 216/72 and does not gain from 224/56.
constexpr int REG_LAUNCH = 168;
// Conditional rescale threshold in log2 units: the running max used for the
// exponentials is only moved when a new row max exceeds it by more than TAU,
// so unnormalised probabilities stay below 2^TAU.  O / l is unchanged by the
// choice because P and l always share the same stale max.
constexpr float TAU = 8.0f;
// 8-bit path: P is stored as e4m3 (largest finite 448, smallest subnormal
// 2^-9).  There the reference max moves when a row max exceeds it by more
// than TAU_FP8, and p is taken as 2^(s - m + P_SHIFT_FP8), so that
// 0 < p <= 2^(TAU_FP8 + P_SHIFT_FP8) = 2^8.75 ~ 430.5 < 448.  Terms below
// 2^-14 of the reference (2^-14 to 2^-17.75 of the row max) underflow to 0;
// l carries the same factor, which O / l cancels and the LSE subtracts.
// The warp-wide O correction runs whenever any of a warp's 32 rows moves its
// reference, so the threshold sets how often it runs.  Against threshold 0
// with a 2^8 scale, threshold 2 (scale 2^6) made the B2/H32/N4096/d128 causal
// 8-bit forward 6.5% faster, 2.75 (2^6) 13%, and 3.75 (2^5) 16%; the error
// against the oracle did not change.
constexpr float TAU_FP8 = 3.75f;
constexpr float P_SHIFT_FP8 = 5.0f;
static_assert(TAU_FP8 + P_SHIFT_FP8 <= 8.75f, "p must stay below the largest finite e4m3 value, 448");
// L2 prefetch of the next unit: issued when the producer starts loading the
// K/V tile PREFETCH_LEAD tiles before the end of the current unit, covering
// the next unit's Q tiles and its first PREFETCH_KV_TILES K/V tiles.
constexpr int PREFETCH_LEAD = 6;
constexpr int PREFETCH_KV_TILES = 3;
// The softmax hands P_t to the issuer in P_PARTS key ranges (1, 2 or 4), so
// that the P V products of one range run while the next is exponentiated.
// Two halves measured best on GB300: against one hand-over, +6% on the
// B2/H32/N4096/d128 causal forward and +7% on GQA N16384; four quarters lose
// the gain again to the extra TMEM store waits and barrier round trips.
#ifndef FA_P_PARTS
#define FA_P_PARTS 2
#endif
constexpr int P_PARTS = FA_P_PARTS;
static_assert(P_PARTS == 1 || P_PARTS == 2 || P_PARTS == 4, "P_PARTS divides the four 32-key chunks");
// Software exponentials: the kernel's SOFT template argument, when non-zero,
// sends one score pair in every SOFT of a tile without a mask through
// exp2_soft2 (FMA/ALU pipes) instead of the MUFU unit.  The library launches
// SOFT = 0 unless fa_debug_soft_exp selects the SOFT_EXP_PERIOD instantiation.
// It stays off by default: on GB300 the MUFU unit runs at about a quarter of
// its peak in this kernel while the softmax warps are bound by instruction
// issue, and moving one pair in 4 (3, 2) to the polynomial made the
// B2/H32/N4096/d128 causal forward 24% (29%, 41%) slower, and the 8-bit
// forward 24% (30%, 40%) slower.  The instantiation kept is the one that
// sends the most exponentials through the polynomial (one pair in 2), so that
// the parity tests cover it as fully as possible.
constexpr int SOFT_EXP_PERIOD = 2;

// Device status word: bit (1 << role) is set when that role gave up waiting;
// bit DEBUG_BIT when a debug build's address check failed.
__device__ int g_fa_status;
constexpr int DEBUG_BIT = 5;

// Debug builds (FA_DEBUG) check every computed TMA coordinate, output row
// and TMEM base column before use.  A failed check sets DEBUG_BIT and the
// access is skipped (a skipped copy then ends in the bounded time-out); it
// never traps.  Release builds compile the checks away.
__device__ __forceinline__ bool dcheck(bool ok) {
#ifdef FA_DEBUG
  if (!ok) atomicOr(&g_fa_status, 1 << DEBUG_BIT);
  return ok;
#else
  (void)ok;
  (void)DEBUG_BIT;
  return true;
#endif
}

// FP8 selects the 8-bit path: e4m3 Q, K and V^T, products of kind f8f6f4.
// PAIR selects the CTA-pair path: two CTAs of a cluster share each product
// (tcgen05 cta_group::2, M = 256), each holding its own 128 query rows of a
// 256-row product tile and half of every K tile (64 keys) and V tile (64 head
// dims), so that a K/V tile is read from L2 once per pair and one instruction
// covers both SMs.
template <int D, bool FP8 = false, bool PAIR = false>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(!PAIR || (D == 128 && !FP8), "the CTA-pair path is built for bf16, d = 128");
  static constexpr int ELEM = FP8 ? 1 : 2;             // bytes per element
  static constexpr int TILE_BYTES = BLOCK_M * D * ELEM;  // one 128 x D tile (a V^T tile, D x 128 keys, likewise)
  // Q and K rows are D * ELEM bytes: 128-byte swizzle column blocks, except
  // the 8-bit d = 64 rows of 64 bytes, which use the 64-byte swizzle.
  static constexpr int ROW_BYTES = D * ELEM;
  static constexpr bool SW64 = ROW_BYTES == 64;
  static constexpr int CHUNKS = SW64 ? 1 : ROW_BYTES / 128;  // swizzle column blocks per Q/K row
  static constexpr int CHUNK_COLS = 128 / ELEM;        // elements per column block
  static constexpr int CHUNK_BYTES = BLOCK_M * 128;    // 16 KB
  static constexpr int QK_SBO = SW64 ? 512 : 1024;     // bytes between 8-row groups of a Q/K tile
  static constexpr int SLOT_BYTES = PAIR ? TILE_BYTES / 2 : TILE_BYTES;  // a pair's CTA holds half a tile
  static constexpr int NS = PAIR ? 10 : (TILE_BYTES == 32768 ? 5 : (TILE_BYTES == 16384 ? 8 : 16));  // ring slots
  static constexpr int QK_KSTEPS = D * ELEM / 32;      // 32 bytes of K per product
  static constexpr int PV_KSTEPS = BLOCK_N * ELEM / 32;
  static constexpr int SMEM_Q = NQT * TILE_BYTES;
  static constexpr int SMEM_RING = NS * SLOT_BYTES;
  static constexpr int CTAS = PAIR ? 2 : 1;            // CTAs sharing one product tile
  static constexpr int TILE_ROWS = CTAS * BLOCK_M;     // query rows of one product tile
  static constexpr int UNIT_ROWS = NQT * TILE_ROWS;    // query rows of one work unit
  static constexpr int REG_SOFTMAX = FP8 ? 224 : 216;
  static constexpr int REG_OTHER = FP8 ? 56 : 72;
  static_assert(8 * REG_SOFTMAX + 4 * REG_OTHER <= 12 * REG_LAUNCH, "register split exceeds the launch pool");
  static_assert(2 * REG_SOFTMAX + REG_OTHER <= 512, "register split exceeds a sub-partition");
  // barriers: full[NS], empty[NS], q_full[2], q_empty[2], s_full[2], p_full[2], o_done[2], drain
  static constexpr int NUM_BARS = 2 * NS + (4 + P_PARTS) * NQT + 1;
  static constexpr int SMEM_BYTES = 1024 + SMEM_Q + SMEM_RING + NUM_BARS * 8 + 16;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

struct Params {
  __nv_bfloat16* o;
  float* lse;
  const int* cu_seqlens;  // null: dense
  int B, Hq, Hkv, Nq, Nk, group;
  float scale_log2;       // scale * log2(e)
  int causal;
  int nqb;                // dense: query units per head = ceil(Nq / 256)
  int num_units;          // dense: B * Hq * nqb; packed: computed on the device
  unsigned long long wait_limit_ns;  // bound on every mbarrier wait
  int fault_inject;       // test hook: 1 = the K/V producer withholds its first fill
  int key_align;          // packed sequences: key tiles start at a multiple of this many tokens (1 or 16)
  // 8-bit path only: per-(batch, head) descale factors of Q [B*Hq], K and V
  // [B*Hkv]; the real inputs are code * descale.
  const float* q_descale;
  const float* k_descale;
  const float* v_descale;
  // Extents, for the debug build's checks: rows per head of the Q and K/V
  // tensor maps, their head counts, and the rows of O and LSE.
  int q_rows, kv_rows, q_heads, kv_heads;
  long long o_rows;
};

__device__ __forceinline__ void checked_load(uint32_t dst, const CUtensorMap* map, const MapExtent& e, uint32_t bar,
                                             int x, int y, int z) {
  if (dcheck(tma_coords_ok(e, x, y, z))) tma_load_3d(dst, map, bar, x, y, z);
}
__device__ __forceinline__ void checked_load_pair(uint32_t dst, const CUtensorMap* map, const MapExtent& e,
                                                  uint32_t bar, int x, int y, int z) {
  if (dcheck(tma_coords_ok(e, x, y, z))) tma_load_3d_pair(dst, map, bar, x, y, z);
}
__device__ __forceinline__ void checked_prefetch(const CUtensorMap* map, const MapExtent& e, int x, int y, int z) {
  if (dcheck(tma_coords_ok(e, x, y, z))) tma_prefetch_l2_3d(map, x, y, z);
}

struct Unit {
  int Lq, Lk;        // sequence lengths (queries, keys)
  int row0;          // first query row of the unit, local to the sequence
  int q_y, k_y;      // TMA row coordinate of the sequence's first token (keys: minus kshift)
  int kshift;        // key tiles start kshift keys before the sequence (8-bit packed path: k_y % 16 == 0)
  int q_z, k_z;      // TMA head coordinate
  long long out_row; // global row index (in O / LSE rows) of the sequence's token 0
};

__device__ __forceinline__ int clampi(int x, int lo, int hi) { return x < lo ? lo : (x > hi ? hi : x); }

// Unit u -> (sequence, head, query block of unit_rows rows).  Dense units are
// ordered longest-first under a causal mask: the last query blocks of every
// head come first, so the persistent CTAs start on the heaviest work.
__device__ __forceinline__ bool decode_unit(const Params& p, int u, Unit& w, int unit_rows) {
  if (p.cu_seqlens == nullptr) {
    const int bh_count = p.B * p.Hq;
    const int qb = p.nqb - 1 - u / bh_count;
    const int bh = u % bh_count;
    const int b = bh / p.Hq, h = bh % p.Hq;
    w.Lq = p.Nq;
    w.Lk = p.Nk;
    w.row0 = qb * unit_rows;
    w.q_y = 0;
    w.k_y = 0;
    w.kshift = 0;
    w.q_z = bh;
    w.k_z = b * p.Hkv + h / p.group;
    w.out_row = static_cast<long long>(bh) * p.Nq;
    return true;
  }
  // Packed sequences: u = blk * Hq + h, blk enumerates every sequence's query
  // blocks in order, the last block of a sequence first.
  const int h = u % p.Hq;
  int blk = u / p.Hq;
  const int T = p.Nq;
  int prev = clampi(__ldg(p.cu_seqlens), 0, T);
  for (int s = 0; s < p.B; ++s) {
    const int next = clampi(__ldg(p.cu_seqlens + s + 1), prev, T);
    const int L = next - prev;
    const int nb = (L + unit_rows - 1) / unit_rows;
    if (blk < nb) {
      w.Lq = L;
      w.Lk = L;
      w.row0 = (nb - 1 - blk) * unit_rows;
      w.q_y = prev;
      // The 8-bit path reads V^T tiles along the token axis, where a TMA box
      // must start on a 16-byte boundary: its key tiles start at the multiple
      // of 16 at or below the sequence start, and the keys before the start
      // are masked.
      w.kshift = prev % p.key_align;
      w.k_y = prev - w.kshift;
      w.q_z = h;
      w.k_z = h / p.group;
      w.out_row = static_cast<long long>(h) * T + prev;
      return true;
    }
    blk -= nb;
    prev = next;
  }
  return false;
}

__device__ __forceinline__ int packed_num_units(const Params& p, int unit_rows) {
  const int T = p.Nq;
  int prev = clampi(__ldg(p.cu_seqlens), 0, T);
  int total = 0;
  for (int s = 0; s < p.B; ++s) {
    const int next = clampi(__ldg(p.cu_seqlens + s + 1), prev, T);
    total += (next - prev + unit_rows - 1) / unit_rows;
    prev = next;
  }
  return total * p.Hq;
}

// Number of K/V tiles product tile t (tile_rows query rows) of unit w must
// visit (0: no key visible to any of its rows).
__device__ __forceinline__ int kv_tiles(const Params& p, const Unit& w, int t, int tile_rows) {
  const int q0 = w.row0 + t * tile_rows;
  if (q0 >= w.Lq || w.Lk <= 0) return 0;
  int last_key = w.Lk - 1;
  if (p.causal) {
    const int last_row = min(q0 + tile_rows - 1, w.Lq - 1);
    last_key = min(last_key, last_row + (w.Lk - w.Lq));
    if (last_key < 0) return 0;
  }
  return (last_key + w.kshift) / BLOCK_N + 1;
}

// Instruction descriptor, kind::f8f6f4 with e4m3 A and B (format code 0),
// fp32 accumulation, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A * B for 8-bit operands (A in shared or tensor memory).
__device__ __forceinline__ void umma_ss_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Four fp32 values to e4m3 (round to nearest even, saturating), x0 in the
// lowest byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float x0, float x1, float x2, float x3) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  return r;
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// The CTA's abort flag and, on the CTA-pair path, the other CTA's flag: a role
// that gives up stops both CTAs of the pair, since each waits on the other.
struct Abort {
  volatile int* flag;
  uint32_t partner;  // cluster address of the other CTA's flag (pair path only)
  bool pair;
  __device__ __forceinline__ void raise(int role) const {
    *flag = 1;
    if (pair) st_cluster_u32(partner, 1u);
    atomicOr(&g_fa_status, 1 << role);
  }
};

// Bounded wait; `cluster` selects acquire semantics at cluster scope (for
// barriers that the other CTA of a pair also signals).
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, const Abort& ab, int role,
                                              uint64_t limit_ns, bool cluster = false) {
  if (cluster ? mbar_wait_cluster(bar, parity, ab.flag, limit_ns) : mbar_wait(bar, parity, ab.flag, limit_ns))
    return true;
  if (!*ab.flag) ab.raise(role);
  return false;
}

// Teardown waits ignore the abort flag: they only wait for copies and MMAs
// that were already issued, which complete on their own.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, const Abort& ab, int role,
                                           uint64_t limit_ns) {
  __shared__ int never;
  never = 0;
  if (!mbar_wait_cluster(bar, parity, &never, limit_ns)) ab.raise(role);
}

template <int D, bool FP8, int SOFT, bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const Params p,
                  const __grid_constant__ SchedTable sc) {
  using C = Cfg<D, FP8, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + C::SMEM_Q;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sRing + C::SMEM_RING);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t bar_base = smem_u32(bars);
  auto full_bar = [&](int s) { return bar_base + 8u * s; };
  auto empty_bar = [&](int s) { return bar_base + 8u * (C::NS + s); };
  auto qfull_bar = [&](int t) { return bar_base + 8u * (2 * C::NS + t); };
  auto qempty_bar = [&](int t) { return bar_base + 8u * (2 * C::NS + NQT + t); };
  auto sfull_bar = [&](int t) { return bar_base + 8u * (2 * C::NS + 2 * NQT + t); };
  auto pfull_bar = [&](int t) { return bar_base + 8u * (2 * C::NS + 3 * NQT + t); };
  auto odone_bar = [&](int t) { return bar_base + 8u * (2 * C::NS + 4 * NQT + t); };
  // ppart_bar(t, i): keys [0, (i + 1) * BLOCK_N / P_PARTS) of P_t are in place (i < P_PARTS - 1).
  auto ppart_bar = [&](int t, int i) { return bar_base + 8u * (2 * C::NS + (5 + i) * NQT + t); };
  const uint32_t drain_bar = bar_base + 8u * (2 * C::NS + (4 + P_PARTS) * NQT);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // Pair path: CTA rank 0 of the cluster issues the products of both CTAs;
  // the full, q_full and P barriers that the issuer waits on live in its
  // shared memory and count the other CTA's copies and arrivals too.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  auto leader_bar = [&](uint32_t bar) { return PAIR ? cluster_addr(bar, 0) : bar; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int t = 0; t < NQT; ++t) {
      mbar_init(qfull_bar(t), 1);
      mbar_init(qempty_bar(t), 1);
      mbar_init(sfull_bar(t), 1);
      mbar_init(pfull_bar(t), C::CTAS * BLOCK_M / 32);  // one arrival per softmax warp of the pair
      for (int i = 0; i + 1 < P_PARTS; ++i) mbar_init(ppart_bar(t, i), C::CTAS * BLOCK_M / 32);
      mbar_init(odone_bar(t), 1);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == WARP_MMA) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), 512);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync_all();  // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{abort_flag, PAIR ? cluster_addr(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u) : 0u, PAIR};
  // Everything above touches only this CTA's shared memory and TMEM, so it
  // overlaps the tail of the previous kernel in the stream; inputs (including
  // cu_seqlens) and outputs are touched only after that kernel is done.  The
  // next kernel may then start its own set-up on the SMs this grid frees.
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  // Map extents for the debug checks.  On the pair path a CTA whose rows lie
  // past the sequence end still loads its (all-fill) Q box, and the odd CTA's
  // half of the last K tile (keys [64, 128)) may start past the last key.
  const MapExtent eq{D, p.q_rows, p.q_heads, C::ELEM, PAIR ? BLOCK_M : 0};
  const MapExtent ek{D, p.kv_rows, p.kv_heads, C::ELEM, PAIR ? BLOCK_N / 2 : 0};
  const MapExtent ev = FP8 ? MapExtent{p.kv_rows, D, p.kv_heads, 1, 0} : ek;  // 8-bit: V^T, keys along x

  const int num_units = (p.cu_seqlens == nullptr) ? p.num_units : packed_num_units(p, C::UNIT_ROWS);
  // Static "snake" schedule over the grid's G persistent workers (CTAs, or
  // CTA pairs on the pair path): in round k the workers take units
  // [k*G, (k+1)*G) in alternating directions, so the longest-first unit list
  // is spread evenly (with the 1:16 cost range of a causal head the busiest
  // worker stays within a few percent of the mean, against 13% for plain
  // round-robin).
  // With a host-built table (dense problems) worker w runs its own list of
  // units instead (SchedTable: head groups visited in turn, longest first).
  const int G = static_cast<int>(gridDim.x) / C::CTAS;
  const int worker = static_cast<int>(blockIdx.x) / C::CTAS;
  const bool table = sc.workers == G && p.cu_seqlens == nullptr;
  const int slot0 = table ? sc.start[worker] : 0;
  const int slots = table ? sc.start[worker + 1] - slot0 : (num_units + G - 1) / G;
  auto snake_unit = [&](int k) {
    return table ? static_cast<int>(sc.unit[slot0 + k]) : k * G + ((k & 1) ? (G - 1 - worker) : worker);
  };
  auto tiles_of = [&](const Unit& w, int t) { return kv_tiles(p, w, t, C::TILE_ROWS); };

  if (warp >= 8) {
  setmaxnreg_dec<C::REG_OTHER>();
  if (warp == WARP_PRODUCER) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      if (p.Nk > 0) {  // with no keys the K/V maps are left unencoded and never used
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
      }
      uint32_t it = 0;
      bool ok = true;
      // The next unit's Q tiles and first K/V tiles usually come from DRAM
      // (another head); warming them into L2 a few K/V tiles before the
      // current unit ends hides most of that latency at the unit boundary.
      auto prefetch_next_unit = [&](int k_next) {
        if (k_next >= slots) return;
        const int un = snake_unit(k_next);
        if (un >= num_units) return;
        Unit wn;
        if (!decode_unit(p, un, wn, C::UNIT_ROWS)) return;
        const int nk0 = tiles_of(wn, 0), nk1 = tiles_of(wn, 1);
        for (int t = 0; t < NQT; ++t) {
          if ((t == 0 ? nk0 : nk1) == 0) continue;
          for (int c = 0; c < C::CHUNKS; ++c)
            checked_prefetch(&tm_q, eq, c * C::CHUNK_COLS, wn.q_y + wn.row0 + t * C::TILE_ROWS + rank * BLOCK_M,
                               wn.q_z);
        }
        const int nn = min(max(nk0, nk1), PREFETCH_KV_TILES);
        for (int j = 0; j < nn; ++j)
          for (int c = 0; c < C::CHUNKS; ++c) {
            if constexpr (PAIR) {  // this CTA's halves: keys [64 rank, +64) of K, columns [64 rank, +64) of V
              checked_prefetch(&tm_k, ek, c * C::CHUNK_COLS, wn.k_y + j * BLOCK_N + rank * (BLOCK_N / 2), wn.k_z);
              if (c == 0) checked_prefetch(&tm_v, ev, rank * C::CHUNK_COLS, wn.k_y + j * BLOCK_N, wn.k_z);
            } else {
              checked_prefetch(&tm_k, ek, c * C::CHUNK_COLS, wn.k_y + j * BLOCK_N, wn.k_z);
              if constexpr (FP8)  // V^T: keys along x, head dims along y
                checked_prefetch(&tm_v, ev, wn.k_y + j * BLOCK_N, 0, wn.k_z);
              else
                checked_prefetch(&tm_v, ev, c * C::CHUNK_COLS, wn.k_y + j * BLOCK_N, wn.k_z);
            }
          }
      };
      for (int k = 0; k < slots && ok; ++k) {
        const int u = snake_unit(k);
        if (u >= num_units) continue;
        Unit w;
        if (!decode_unit(p, u, w, C::UNIT_ROWS)) continue;
        const int nmax = max(tiles_of(w, 0), tiles_of(w, 1));
        if (nmax <= PREFETCH_LEAD) prefetch_next_unit(k + 1);
        for (int j = 0; j < nmax && ok; ++j) {
          if (j == nmax - PREFETCH_LEAD) prefetch_next_unit(k + 1);
          for (int kv = 0; kv < 2; ++kv) {
            const int s = it % C::NS;
            if (!(ok = wait_or_abort(empty_bar(s), ((it / C::NS) & 1u) ^ 1u, ab, 0, p.wait_limit_ns, PAIR))) break;
            if (p.fault_inject == 1 && it == 0) {  // test hook: this fill never arrives
              ++it;
              continue;
            }
            const uint32_t dst = smem_u32(sRing + s * C::SLOT_BYTES);
            if constexpr (PAIR) {
              // Both CTAs' halves are counted on the even CTA's full barrier,
              // which that CTA arms for the whole tile.
              const uint32_t fb = leader_bar(full_bar(s));
              if (rank == 0) mbar_arrive_expect_tx(full_bar(s), 2 * C::SLOT_BYTES);
              if (kv == 0) {  // K: keys [64 rank, +64) of the tile, every head dim
                for (int c = 0; c < C::CHUNKS; ++c)
                  checked_load_pair(dst + c * (C::SLOT_BYTES / C::CHUNKS), &tm_k, ek, fb, c * C::CHUNK_COLS,
                                    w.k_y + j * BLOCK_N + rank * (BLOCK_N / 2), w.k_z);
              } else {        // V: head dims [64 rank, +64) of every key of the tile
                checked_load_pair(dst, &tm_v, ev, fb, rank * C::CHUNK_COLS, w.k_y + j * BLOCK_N, w.k_z);
              }
            } else {
              mbar_arrive_expect_tx(full_bar(s), C::TILE_BYTES);
              if (FP8 && kv) {  // V^T tile: 128 head dims (rows) x 128 keys (bytes)
                checked_load(dst, &tm_v, ev, full_bar(s), w.k_y + j * BLOCK_N, 0, w.k_z);
              } else {
                for (int c = 0; c < C::CHUNKS; ++c)
                  checked_load(dst + c * C::CHUNK_BYTES, kv ? &tm_v : &tm_k, kv ? ev : ek, full_bar(s),
                               c * C::CHUNK_COLS, w.k_y + j * BLOCK_N, w.k_z);
              }
            }
            ++it;
          }
        }
      }
      // Wait until every issued copy has landed before the CTA may exit.  On
      // the pair path the even CTA's full barriers count both CTAs' copies;
      // the odd CTA cannot observe them and relies on the teardown below.
      if (!PAIR || rank == 0) {
        for (int s = 0; s < C::NS; ++s) {
          if (it > static_cast<uint32_t>(s)) {
            const uint32_t f = s + C::NS * ((it - 1 - s) / C::NS);
            wait_drain(full_bar(s), (f / C::NS) & 1u, ab, 0, p.wait_limit_ns);
          }
        }
      }
    }
  } else if (warp == WARP_QLOAD) {
    // ------------------------------------------------------------- Q loads
    if (lane == 0) {
      uint32_t qfills[NQT] = {0, 0};
      bool ok = true;
      for (int k = 0; k < slots && ok; ++k) {
        const int u = snake_unit(k);
        if (u >= num_units) continue;
        Unit w;
        if (!decode_unit(p, u, w, C::UNIT_ROWS)) continue;
#pragma unroll
        for (int t = 0; t < NQT; ++t) {
          if (!ok || tiles_of(w, t) == 0) continue;
          if (!(ok = wait_or_abort(qempty_bar(t), (qfills[t] & 1u) ^ 1u, ab, 4, p.wait_limit_ns, PAIR))) continue;
          const uint32_t dst = smem_u32(sQ + t * C::TILE_BYTES);
          const int row = w.q_y + w.row0 + t * C::TILE_ROWS + static_cast<int>(rank) * BLOCK_M;
          if constexpr (PAIR) {
            if (rank == 0) mbar_arrive_expect_tx(qfull_bar(t), 2 * C::TILE_BYTES);
            for (int c = 0; c < C::CHUNKS; ++c)
              checked_load_pair(dst + c * C::CHUNK_BYTES, &tm_q, eq, leader_bar(qfull_bar(t)), c * C::CHUNK_COLS,
                                row, w.q_z);
          } else {
            mbar_arrive_expect_tx(qfull_bar(t), C::TILE_BYTES);
            for (int c = 0; c < C::CHUNKS; ++c)
              checked_load(dst + c * C::CHUNK_BYTES, &tm_q, eq, qfull_bar(t), c * C::CHUNK_COLS, row, w.q_z);
          }
          ++qfills[t];
        }
      }
      if (!PAIR || rank == 0) {
#pragma unroll
        for (int t = 0; t < NQT; ++t)
          if (qfills[t] > 0) wait_drain(qfull_bar(t), (qfills[t] - 1) & 1u, ab, 4, p.wait_limit_ns);
      }
    }
  } else if (warp == WARP_MMA && (!PAIR || rank == 0)) {
    // ------------------------------------------------------------------ MMA
    // Per tile the order is QK(0), then for each j: PV(j), QK(j+1); S_t is
    // therefore overwritten by QK(j+1) only after PV(j) has read the P that
    // aliases it (the products of one thread complete in issue order).
    uint32_t elected;
    asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}" : "=r"(elected));
    const bool leader = elected != 0;
    // 8-bit path: both products K-major (V arrives transposed), 32 bytes of K each.
    constexpr uint32_t IDESC_QK =
        FP8 ? idesc_e4m3_f32(BLOCK_M, BLOCK_N) : idesc_bf16_f32(C::TILE_ROWS, BLOCK_N, 0, 0);
    constexpr uint32_t IDESC_PV = FP8 ? idesc_e4m3_f32(BLOCK_M, D) : idesc_bf16_f32(C::TILE_ROWS, D, 0, 1);
    const uint32_t q_addr = smem_u32(sQ);
    const uint32_t ring_addr = smem_u32(sRing);
    // Byte stride between the 128-byte-wide column blocks of a K slot: a full
    // 128-row tile, or the 64-key half a CTA of a pair holds.
    constexpr int K_CHUNK_BYTES = C::SLOT_BYTES / C::CHUNKS;
    // S_t = Q_t K^T: both operands K-major (head dim contiguous), 16 columns per MMA.
    auto qk_desc = [&](uint32_t addr) {
      return C::SW64 ? smem_desc_sw64(addr, 16, C::QK_SBO) : smem_desc_sw128(addr, 16, C::QK_SBO);
    };
    auto issue_qk = [&](int t, int slot) {
      const uint64_t q_desc = qk_desc(q_addr + t * C::TILE_BYTES);
      const uint64_t k_desc = qk_desc(ring_addr + slot * C::SLOT_BYTES);
#pragma unroll
      for (int kk = 0; kk < C::QK_KSTEPS; ++kk) {
        const uint64_t qoff = static_cast<uint64_t>((kk / 4) * C::CHUNK_BYTES + (kk % 4) * 32) >> 4;
        const uint64_t koff = static_cast<uint64_t>((kk / 4) * K_CHUNK_BYTES + (kk % 4) * 32) >> 4;
        if (leader) {
          if constexpr (FP8)
            umma_ss_f8(tmem + t * 128, q_desc + qoff, k_desc + koff, IDESC_QK, kk > 0 ? 1u : 0u);
          else if constexpr (PAIR)
            umma_ss_pair(tmem + t * 128, q_desc + qoff, k_desc + koff, IDESC_QK, kk > 0 ? 1u : 0u);
          else
            umma_ss(tmem + t * 128, q_desc + qoff, k_desc + koff, IDESC_QK, kk > 0 ? 1u : 0u);
        }
      }
    };
    // O_t (+)= P_t V: P from TMEM (bf16 pairs), V MN-major (head dim contiguous), 16 keys per MMA.
    auto issue_pv = [&](int t, int slot, bool accumulate, int part) {
      if constexpr (FP8) {
        // V^T K-major (keys contiguous); P as packed e4m3 in TMEM, 8 columns per 32 keys.
        const uint64_t vt_desc = smem_desc_sw128(ring_addr + slot * C::SLOT_BYTES, 16, 1024);
#pragma unroll
        for (int kk = part * C::PV_KSTEPS / P_PARTS; kk < (part + 1) * C::PV_KSTEPS / P_PARTS; ++kk) {
          if (leader)
            umma_ts_f8(tmem + 256 + t * 128, tmem + t * 128 + kk * 8, vt_desc + static_cast<uint64_t>(kk * 32 >> 4),
                       IDESC_PV, (accumulate || kk > 0) ? 1u : 0u);
        }
      } else {
        // On the pair path each CTA's slot holds one 128-byte column block
        // (64 head dims) of V; the stride between blocks is then unused.
        const uint64_t v_desc = smem_desc_sw128(ring_addr + slot * C::SLOT_BYTES, C::CHUNK_BYTES, 1024);
#pragma unroll
        for (int kk = part * BLOCK_N / (16 * P_PARTS); kk < (part + 1) * BLOCK_N / (16 * P_PARTS); ++kk) {
          if (leader) {
            if constexpr (PAIR)
              umma_ts_pair(tmem + 256 + t * 128, tmem + t * 128 + kk * 8,
                           v_desc + static_cast<uint64_t>(kk * 16 * 128 >> 4), IDESC_PV,
                           (accumulate || kk > 0) ? 1u : 0u);
            else
              umma_ts(tmem + 256 + t * 128, tmem + t * 128 + kk * 8,
                      v_desc + static_cast<uint64_t>(kk * 16 * 128 >> 4), IDESC_PV, (accumulate || kk > 0) ? 1u : 0u);
          }
        }
      }
    };
    // Signals a barrier that both CTAs of a pair wait on (the same barrier in
    // each CTA), or the CTA's own barrier.
    auto commit = [&](uint32_t bar) {
      if (leader) {
        if constexpr (PAIR) {
          umma_commit_pair(bar);
          umma_commit_pair(cluster_addr(bar, 1));
        } else {
          umma_commit(bar);
        }
      }
      __syncwarp();
    };
    uint32_t it = 0;
    uint32_t qcnt[NQT] = {0, 0}, pcnt[NQT] = {0, 0};
    bool ok = true;
    for (int k = 0; k < slots && ok; ++k) {
      const int u = snake_unit(k);
      if (u >= num_units) continue;
      Unit w;
      if (!decode_unit(p, u, w, C::UNIT_ROWS)) continue;
      int nkv[NQT];
      int nmax = 0;
#pragma unroll
      for (int t = 0; t < NQT; ++t) {
        nkv[t] = tiles_of(w, t);
        nmax = max(nmax, nkv[t]);
      }
      if (nmax == 0) continue;
#pragma unroll
      for (int t = 0; t < NQT; ++t) {
        if (!ok || nkv[t] == 0) continue;
        ok = wait_or_abort(qfull_bar(t), qcnt[t] & 1u, ab, 1, p.wait_limit_ns, PAIR);
        ++qcnt[t];
      }
      if (!ok) break;
      // K_0 for every active tile.
      {
        const int s = it % C::NS;
        if (!(ok = wait_or_abort(full_bar(s), (it / C::NS) & 1u, ab, 1, p.wait_limit_ns, PAIR))) break;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < NQT; ++t) {
          if (nkv[t] == 0) continue;
          issue_qk(t, s);
          commit(sfull_bar(t));
          if (nkv[t] == 1) commit(qempty_bar(t));
        }
        commit(empty_bar(s));
        ++it;
      }
      for (int j = 0; j < nmax && ok; ++j) {
        const int sv = it % C::NS;
        if (!(ok = wait_or_abort(full_bar(sv), (it / C::NS) & 1u, ab, 1, p.wait_limit_ns, PAIR))) break;
        tc_fence_after();
        ++it;
        const bool has_next = j + 1 < nmax;
        const int sk = it % C::NS;
        bool k_ready = false;
#pragma unroll
        for (int t = 0; t < NQT; ++t) {
          if (!ok || j >= nkv[t]) continue;
          // P_t arrives in P_PARTS key ranges; the products of one range run
          // while the softmax exponentiates the next.
#pragma unroll
          for (int i = 0; i < P_PARTS && ok; ++i) {
            const uint32_t bar = (i + 1 < P_PARTS) ? ppart_bar(t, i) : pfull_bar(t);
            if (!(ok = wait_or_abort(bar, pcnt[t] & 1u, ab, 1, p.wait_limit_ns, PAIR))) break;
            tc_fence_after();
            issue_pv(t, sv, j > 0 || i > 0, i);
          }
          if (!ok) continue;
          ++pcnt[t];
          if (j + 1 == nkv[t]) commit(odone_bar(t));  // last PV of this tile in the unit
          if (j + 1 < nkv[t]) {
            if (!k_ready) {
              if (!(ok = wait_or_abort(full_bar(sk), (it / C::NS) & 1u, ab, 1, p.wait_limit_ns, PAIR))) continue;
              tc_fence_after();
              k_ready = true;
            }
            issue_qk(t, sk);
            commit(sfull_bar(t));
            if (j + 2 == nkv[t]) commit(qempty_bar(t));
          }
        }
        if (!ok) break;
        commit(empty_bar(sv));
        if (has_next) {
          commit(empty_bar(sk));
          ++it;
        }
      }
    }
    // Every MMA issued so far completes before the CTA may release TMEM.
    if (leader) {
      if constexpr (PAIR)
        umma_commit_pair(drain_bar);
      else
        umma_commit(drain_bar);
    }
    __syncwarp();
    wait_drain(drain_bar, 0, ab, 1, p.wait_limit_ns);
  }
  } else {
    setmaxnreg_inc<C::REG_SOFTMAX>();
    // -------------------------------------------------------------- softmax
    const int t = warp / 4;
    const int r = threadIdx.x % 128;
    const uint32_t lane_base = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * 128;
    const uint32_t tO = tmem + lane_base + 256 + t * 128;
    // Debug build: this thread's S and O columns lie inside the 512 allocated.
    dcheck(((tS & 0xFFFFu) - (tmem & 0xFFFFu)) + BLOCK_N <= 512u && ((tO & 0xFFFFu) - (tmem & 0xFFFFu)) + D <= 512u &&
           (tS >> 16) == static_cast<uint32_t>((warp % 4) * 32));
    const float sl2_base = p.scale_log2;
    const float NEG_INF = -INFINITY;
    constexpr float tau = FP8 ? TAU_FP8 : TAU;
    constexpr float p_shift = FP8 ? P_SHIFT_FP8 : 0.f;
    // One arrival per warp on a P barrier of the issuing CTA.  On the pair
    // path the arrival is relaxed: the data it announces is in TMEM, complete
    // once tcgen05.wait::st returns and ordered by tcgen05.fence::before_thread_sync,
    // and no shared- or global-memory write has to be released with it.  A
    // release at cluster scope measured about 900 cycles per arrival on GB300
    // (against about 50), which doubled the softmax's time per K/V tile.
    auto arrive_p = [&](uint32_t bar) {
      if constexpr (PAIR)
        mbar_arrive_remote_relaxed(leader_bar(bar));
      else
        mbar_arrive(bar);
    };
    uint32_t scnt = 0, ocnt = 0;
    bool ok = true;
    for (int k = 0; k < slots && ok; ++k) {
      const int u = snake_unit(k);
      if (u >= num_units) continue;
      Unit w;
      if (!decode_unit(p, u, w, C::UNIT_ROWS)) continue;
      // This CTA's 128 rows of product tile t.
      const int q0 = w.row0 + t * C::TILE_ROWS + static_cast<int>(rank) * BLOCK_M;
      const int nkv = tiles_of(w, t);
      // On the pair path a CTA whose rows all lie past the sequence end still
      // takes part in the tile's steps (the products are shared); it stores nothing.
      if (q0 >= w.Lq && (!PAIR || nkv == 0)) continue;
      const int row = q0 + r;
      const bool row_ok = row < w.Lq;
      const int diag = row + (w.Lk - w.Lq);  // last visible key under the causal mask
      const int tile_diag = q0 + (w.Lk - w.Lq);
      // 8-bit path: the Q and K descales scale every score of this unit.
      float sl2 = sl2_base;
      if constexpr (FP8) sl2 *= __ldg(p.q_descale + w.q_z) * __ldg(p.k_descale + w.k_z);
      float m_used = NEG_INF;
      float l = 0.f;
      for (int j = 0; j < nkv; ++j) {
        if (!(ok = wait_or_abort(sfull_bar(t), scnt & 1u, ab, 2 + t, p.wait_limit_ns, PAIR))) break;
        ++scnt;
        tc_fence_after();
        float s[BLOCK_N];
        {
          uint32_t raw[BLOCK_N];
          tmem_ld128_wait(tS, raw);
#pragma unroll
          for (int i = 0; i < BLOCK_N; ++i) s[i] = __uint_as_float(raw[i]);
        }
        // Key of column 0; on the 8-bit packed path the first tile of a
        // sequence starts up to 15 keys early (columns of the previous sequence).
        const int k0 = j * BLOCK_N - (FP8 ? w.kshift : 0);
        const bool need_mask = (FP8 && k0 < 0) || (k0 + BLOCK_N > w.Lk) || (p.causal && k0 + BLOCK_N - 1 > tile_diag);
        // Column c of this row is visible iff c <= rel (one compare against a
        // constant per element).  rel_hi, the warp's largest limit, lets the
        // exponential loop below skip 32-column chunks no lane can see.
        int rel_hi = BLOCK_N;
        if (need_mask) {
          const int lim = p.causal ? min(w.Lk - 1, diag) : (w.Lk - 1);
          const int rel = lim - k0;
          rel_hi = __reduce_max_sync(0xffffffffu, rel);
#pragma unroll
          for (int c = 0; c < BLOCK_N; ++c)
            if (c > rel) s[c] = NEG_INF;
          if constexpr (FP8) {
#pragma unroll
            for (int c = 0; c < BLOCK_N; ++c)
              if (c < -k0) s[c] = NEG_INF;
          }
        }
        // Row max: 3-input max in 4 independent chains.
        float mx4[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
#pragma unroll
        for (int c = 0; c < BLOCK_N; c += 8) {
#pragma unroll
          for (int i = 0; i < 4; ++i) mx4[i] = max3(mx4[i], s[c + 2 * i], s[c + 2 * i + 1]);
        }
        const float mx = max3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
        const float m_tile = mx * sl2;
        const float m_new = fmaxf(m_used, m_tile);
        const bool need = m_new > m_used + tau;
        if (j == 0) {
          m_used = m_new;
        } else if (__any_sync(0xffffffffu, need)) {
          // PV_t(j-1) was issued before QK_t(j), so the completed s_full phase
          // above already covers it: O is stable here.
          const float alpha = need ? ex2_approx(m_used - m_new) : 1.f;
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t raw[32];
            tmem_ld32_wait(tO + c0, raw);
#pragma unroll
            for (int i = 0; i < 32; ++i) raw[i] = __float_as_uint(__uint_as_float(raw[i]) * alpha);
            tmem_st32(tO + c0, raw);
          }
          l *= alpha;
          if (need) m_used = m_new;
        }
        const float neg_base = (m_used == NEG_INF) ? 0.f : p_shift - m_used;
        // p = 2^(s * scale * log2e - m_used), two scores per packed FMA; the
        // row sum runs in four packed accumulators.
        const float2 c2 = make_float2(sl2, sl2);
        const float2 nb2 = make_float2(neg_base, neg_base);
        float2 acc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c0 = 0; c0 < BLOCK_N; c0 += 32) {
          uint32_t pk[16];   // bf16 pairs
          uint32_t pk8[8];   // 8-bit path: e4m3 quads
          if (c0 > rel_hi) {  // hidden from every lane of the warp: P = 0
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = 0u;
#pragma unroll
            for (int i = 0; i < 8; ++i) pk8[i] = 0u;
          } else {
            float2 prev = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 x = fma2(make_float2(s[c0 + 2 * i], s[c0 + 2 * i + 1]), c2, nb2);
              float2 e;
              if (SOFT > 0 && (i % (SOFT > 0 ? SOFT : 1)) == SOFT - 1 && !need_mask)
                e = exp2_soft2(x);  // no -inf here: the tile has no masked score
              else
                e = make_float2(ex2_approx(x.x), ex2_approx(x.y));
              acc[i % 4] = add2(acc[i % 4], e);
              if constexpr (FP8) {
                if (i & 1) pk8[i / 2] = pack_e4m3x4(prev.x, prev.y, e.x, e.y);
                prev = e;
              } else {
                pk[i] = pack_bf16x2(e.x, e.y);
              }
            }
          }
          if constexpr (FP8)
            tmem_st8(tS + c0 / 4, pk8);
          else
            tmem_st16(tS + c0 / 2, pk);
          constexpr int CHUNKS_PER_PART = BLOCK_N / 32 / P_PARTS;
          if ((c0 / 32 + 1) % CHUNKS_PER_PART == 0 && c0 + 32 < BLOCK_N) {  // a key range of P is in place
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_p(ppart_bar(t, c0 / 32 / CHUNKS_PER_PART));
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_p(pfull_bar(t));
        {
          const float2 a01 = add2(acc[0], acc[1]);
          const float2 a23 = add2(acc[2], acc[3]);
          const float2 a = add2(a01, a23);
          l += a.x + a.y;
        }
      }
      if (!ok) break;
      // ------------------------------------------------------------ epilogue
      if (nkv > 0) {
        if (!(ok = wait_or_abort(odone_bar(t), ocnt & 1u, ab, 2 + t, p.wait_limit_ns, PAIR))) break;
        ++ocnt;
        tc_fence_after();
      }
      float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      if constexpr (FP8) inv_l *= __ldg(p.v_descale + w.k_z);
      __nv_bfloat16* orow = p.o + (w.out_row + row) * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t raw[32];
        if (nkv > 0) {
          tmem_ld32_wait(tO + c0, raw);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) raw[i] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(raw[2 * i]) * inv_l, __uint_as_float(raw[2 * i + 1]) * inv_l);
        if (row_ok && dcheck(w.out_row + row >= 0 && w.out_row + row < p.o_rows)) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if (row_ok && dcheck(w.out_row + row >= 0 && w.out_row + row < p.o_rows)) {
        const float lse = (l > 0.f) ? (m_used - p_shift + __log2f(l)) * 0.69314718055994531f : NEG_INF;
        p.lse[w.out_row + row] = lse;
      }
    }
  }

  // -------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) {
    // The products of the even CTA read the odd CTA's shared memory and write
    // its TMEM, and the odd CTA's copies are counted in the even CTA's
    // barriers: neither CTA leaves (or frees TMEM) before the other is done.
    // After a time-out, copies issued by the odd CTA that the even CTA no
    // longer waits for are given a fixed 0.5 ms to land first.
    cluster_sync_all();
    if (*abort_flag && threadIdx.x == 0) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 500000ull) {
      }
    }
    __syncthreads();
    cluster_sync_all();
  }
  if (warp == WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem, 512);
    else
      tmem_dealloc(tmem, 512);
  }
}

// Applies exp2_soft2 to pairs of x (test entry point for its error bound).
__global__ void exp2_soft_kernel(const float* __restrict__ x, float* __restrict__ y, int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i + 1 < n) {
    const float2 r = exp2_soft2(make_float2(x[i], x[i + 1]));
    y[i] = r.x;
    y[i + 1] = r.y;
  } else if (i < n) {
    y[i] = exp2_soft2(make_float2(x[i], 0.f)).x;
  }
}

// ============================================================================
// Host side
// ============================================================================

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult qres;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qres) ==
            cudaSuccess &&
        qres == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// [heads, rows, d] bf16 tensor, loaded as box_rows x 64-column boxes with the
// 128-byte swizzle that the UMMA K-major / MN-major descriptors expect.
bool encode_bf16_rows_map(CUtensorMap* map, const void* base, int d, long long rows, long long heads, int box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(rows) * d * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t elem[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool encode_rows_map(CUtensorMap* map, const void* base, int d, long long rows, long long heads) {
  return encode_bf16_rows_map(map, base, d, rows, heads, BLOCK_M);
}

// Raises the dynamic shared-memory limit of one kernel instantiation, once
// per device (the attribute applies to the current device).  For the
// CTA-pair instantiation it also finds how many CTA pairs can be resident at
// once (*pairs); 0 if none.
template <int D, bool FP8, int SOFT, bool PAIR>
static bool prepare_kernel(int device, int* pairs = nullptr) {
  static std::mutex mu;
  static bool attr_set[kMaxDevicesDecode] = {};
  static int max_pairs[kMaxDevicesDecode] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= kMaxDevicesDecode) return false;
  if (!attr_set[device]) {
    if (cudaFuncSetAttribute(fa_fwd_kernel<D, FP8, SOFT, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<D, FP8, PAIR>::SMEM_BYTES) != cudaSuccess)
      return false;
    if (PAIR) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2, 1, 1);
      cfg.blockDim = dim3(NUM_THREADS, 1, 1);
      cfg.dynamicSmemBytes = Cfg<D, FP8, PAIR>::SMEM_BYTES;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, fa_fwd_kernel<D, FP8, SOFT, PAIR>, &cfg) != cudaSuccess) return false;
      max_pairs[device] = n;
    }
    attr_set[device] = true;
  }
  if (pairs) *pairs = max_pairs[device];
  return true;
}

// Launches one instantiation on `stream` (programmatic stream serialization,
// see PdlLaunch) as `clusters` clusters of `cta_per` CTAs.
template <typename Kernel>
static fa_status launch_kernel(Kernel kernel, long long clusters, int cta_per, int smem, cudaStream_t stream,
                               const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const Params& prm,
                               const SchedTable& sc) {
  PdlLaunch L(dim3(static_cast<unsigned>(clusters * cta_per)), NUM_THREADS, smem, stream, static_cast<unsigned>(cta_per));
  return cudaLaunchKernelEx(&L.cfg, kernel, tq, tk, tv, prm, sc) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// The schedule builder's view of a dense forward unit (decode_unit's order):
// cost = K/V steps of its longer query tile plus two steps of per-unit
// overhead (Q wait, first K/V wait, epilogue; 2 to 2.5 measured about 1%
// faster than 1 on the B2/H32/N4096 causal workload, 4 slower); group = its
// KV head's group.
struct FwdSchedCtx {
  int B, Hq, Hkv, Nq, Nk, causal, unit_rows, tile_rows, nqb, group_heads;
};

static void describe_fwd_unit(const void* vctx, int u, SchedUnit* out) {
  const FwdSchedCtx& c = *static_cast<const FwdSchedCtx*>(vctx);
  const int bh_count = c.B * c.Hq;
  const int qb = c.nqb - 1 - u / bh_count;
  const int bh = u % bh_count;
  const int kv_head = (bh / c.Hq) * c.Hkv + (bh % c.Hq) / (c.Hq / c.Hkv);
  int steps = 0;
  for (int t = 0; t * c.tile_rows < c.unit_rows; ++t) {
    const int q0 = qb * c.unit_rows + t * c.tile_rows;
    if (q0 >= c.Nq || c.Nk <= 0) continue;
    int last_key = c.Nk - 1;
    if (c.causal) last_key = std::min(last_key, std::min(q0 + c.tile_rows - 1, c.Nq - 1) + (c.Nk - c.Nq));
    if (last_key >= 0) steps = std::max(steps, last_key / BLOCK_N + 1);
  }
  out->cost = static_cast<float>(steps) + 2.0f;
  out->group = kv_head / c.group_heads;
}

// Table for a dense single-CTA launch of `grid` workers (workers = 0: snake).
static void fwd_schedule(SchedTable* sc, int kind, int B, int Hq, int Hkv, int Nq, int Nk, int D, int elem_bytes,
                         int causal, int unit_rows, int nqb, long long units, long long grid) {
  sc->workers = 0;
  if (units > kSchedCap || grid > kSchedMaxWorkers || units <= grid) return;
  FwdSchedCtx c{B, Hq, Hkv, Nq, Nk, causal, unit_rows, BLOCK_M, nqb,
                sched_group_heads(2.0 * static_cast<double>(Nk) * D * elem_bytes)};
  const long long key[12] = {kind, B, Hq, Hkv, Nq, Nk, D, causal, unit_rows, grid, elem_bytes, 0};
  build_schedule(key, static_cast<int>(grid), static_cast<int>(units), describe_fwd_unit, &c, sc);
}

// Tensor extents for the debug build's checks (tensor-map heads: (batch,
// head) pairs, or heads alone when packed).
static void set_extents(Params& prm, long long q_heads, long long kv_heads) {
  prm.q_rows = prm.Nq;
  prm.kv_rows = prm.Nk;
  prm.q_heads = static_cast<int>(q_heads);
  prm.kv_heads = static_cast<int>(kv_heads);
  prm.o_rows = q_heads * prm.Nq;
}

template <int D>
static fa_status launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int Nq, int Nk, float scale, int causal, const int32_t* cu_seqlens, cudaStream_t stream,
                        const LaunchEnv& env) {
  if (decode_supported(B, Hq, Hkv, Nq, Nk, D, cu_seqlens))
    return launch_decode(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, stream, env.sms, env.wait_limit_ns,
                         env.fault_mode);
  const bool soft = env.soft_exp != 0;
  // The CTA-pair kernel runs bf16 problems with d = 128 only when the
  // fa_debug_fwd_pair hook selects it: on GB300 it measured slower than the
  // single-CTA kernel (the step is set by the MMA issuer and the per-tile
  // softmax chain, and a pair has one issuer for two SMs).
  int pairs = 0;
  bool pair = false;
  if constexpr (D == 128) {
    if (env.fwd_pair && !soft) {
      if (!prepare_kernel<D, false, 0, true>(env.device, &pairs)) return FA_ERR_CUDA;
      pair = pairs > 0;
    }
  }
  if (!pair && !(soft ? prepare_kernel<D, false, SOFT_EXP_PERIOD, false>(env.device)
                      : prepare_kernel<D, false, 0, false>(env.device)))
    return FA_ERR_CUDA;
  const bool packed = cu_seqlens != nullptr;
  const long long q_heads = packed ? Hq : static_cast<long long>(B) * Hq;
  const long long kv_heads = packed ? Hkv : static_cast<long long>(B) * Hkv;
  alignas(64) CUtensorMap tq, tk, tv;
  std::memset(&tq, 0, sizeof(tq));
  std::memset(&tk, 0, sizeof(tk));
  std::memset(&tv, 0, sizeof(tv));
  if (!encode_rows_map(&tq, q, D, Nq, q_heads)) return FA_ERR_CUDA;
  // A CTA of a pair loads 64-key halves of K tiles.
  if (Nk > 0 && (!encode_bf16_rows_map(&tk, k, D, Nk, kv_heads, pair ? BLOCK_N / 2 : BLOCK_N) ||
                 !encode_rows_map(&tv, v, D, Nk, kv_heads)))
    return FA_ERR_CUDA;
  const int unit_rows = (pair ? 2 : 1) * NQT * BLOCK_M;  // Cfg<D, false, pair>::UNIT_ROWS
  const long long workers = pair ? pairs : env.sms;
  Params prm;
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.cu_seqlens = cu_seqlens;
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Nq = Nq;
  prm.Nk = Nk;
  prm.group = Hq / Hkv;
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  prm.causal = causal ? 1 : 0;
  prm.wait_limit_ns = env.wait_limit_ns;
  prm.fault_inject = env.fault_mode == kFaultFwd ? 1 : 0;
  prm.key_align = 1;
  prm.q_descale = prm.k_descale = prm.v_descale = nullptr;
  set_extents(prm, q_heads, kv_heads);
  long long grid;  // persistent workers: CTAs, or CTA pairs
  if (packed) {
    prm.nqb = 0;
    prm.num_units = -1;
    // Upper bound on units: every sequence adds at most one partial block.
    const long long bound = static_cast<long long>(Hq) * ((Nq + unit_rows - 1) / unit_rows + B);
    grid = bound < workers ? bound : workers;
  } else {
    prm.nqb = (Nq + unit_rows - 1) / unit_rows;
    const long long units = static_cast<long long>(B) * Hq * prm.nqb;
    if (units > 0x7fffffffLL) return FA_ERR_SHAPE;
    prm.num_units = static_cast<int>(units);
    grid = units < workers ? units : workers;
  }
  if (grid <= 0) return FA_OK;
  SchedTable sc;
  sc.workers = 0;
  if (!packed && !pair)
    fwd_schedule(&sc, 0, B, Hq, Hkv, Nq, Nk, D, 2, prm.causal, unit_rows, prm.nqb, prm.num_units, grid);
  if constexpr (D == 128) {
    if (pair)
      return launch_kernel(fa_fwd_kernel<D, false, 0, true>, grid, 2, Cfg<D, false, true>::SMEM_BYTES, stream, tq,
                           tk, tv, prm, sc);
  }
  if (soft)
    return launch_kernel(fa_fwd_kernel<D, false, SOFT_EXP_PERIOD, false>, grid, 1, Cfg<D>::SMEM_BYTES, stream, tq, tk,
                         tv, prm, sc);
  return launch_kernel(fa_fwd_kernel<D, false, 0, false>, grid, 1, Cfg<D>::SMEM_BYTES, stream, tq, tk, tv, prm, sc);
}

fa_status launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                     int Nq, int Nk, int d, float scale, int causal, const int32_t* cu_seqlens, cudaStream_t stream,
                     const LaunchEnv& env) {
  if (d == 128) return launch<128>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, cu_seqlens, stream, env);
  return launch<64>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, cu_seqlens, stream, env);
}

// [heads, rows, cols] uint8 tensor read in box_rows x box_cols boxes with the
// 128-byte swizzle (box_cols = 128) or the 64-byte swizzle (box_cols = 64):
// the K-major layout of an 8-bit operand tile.
static bool encode_u8_map(CUtensorMap* map, const void* base, long long cols, long long rows, long long heads,
                          int box_cols, int box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows * cols)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t elem[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
static fa_status launch_fp8(const void* q8, const void* k8, const void* vt8, const float* q_descale,
                            const float* k_descale, const float* v_descale, void* o, float* lse, int B, int Hq,
                            int Hkv, int Nq, int Nk, float scale, int causal, const int32_t* cu_seqlens,
                            cudaStream_t stream, const LaunchEnv& env) {
  using C = Cfg<D, true>;
  const bool soft = env.soft_exp != 0;
  if (!(soft ? prepare_kernel<D, true, SOFT_EXP_PERIOD, false>(env.device)
             : prepare_kernel<D, true, 0, false>(env.device)))
    return FA_ERR_CUDA;
  const bool packed = cu_seqlens != nullptr;
  const long long q_heads = packed ? Hq : static_cast<long long>(B) * Hq;
  const long long kv_heads = packed ? Hkv : static_cast<long long>(B) * Hkv;
  alignas(64) CUtensorMap tq, tk, tv;
  std::memset(&tk, 0, sizeof(tk));
  std::memset(&tv, 0, sizeof(tv));
  // Q and K: rows of D bytes (one swizzle block); V^T: D rows of Nk bytes, read in 128-key boxes.
  if (!encode_u8_map(&tq, q8, D, Nq, q_heads, C::ROW_BYTES, BLOCK_M)) return FA_ERR_CUDA;
  if (Nk > 0 && (!encode_u8_map(&tk, k8, D, Nk, kv_heads, C::ROW_BYTES, BLOCK_M) ||
                 !encode_u8_map(&tv, vt8, Nk, D, kv_heads, BLOCK_N, D)))
    return FA_ERR_CUDA;
  Params prm;
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.cu_seqlens = cu_seqlens;
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.Nq = Nq;
  prm.Nk = Nk;
  prm.group = Hq / Hkv;
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  prm.causal = causal ? 1 : 0;
  prm.wait_limit_ns = env.wait_limit_ns;
  prm.fault_inject = 0;
  prm.key_align = packed ? 16 : 1;  // V^T boxes start on 16-byte (16-key) boundaries
  prm.q_descale = q_descale;
  prm.k_descale = k_descale;
  prm.v_descale = v_descale;
  set_extents(prm, q_heads, kv_heads);
  long long grid;
  if (packed) {
    prm.nqb = 0;
    prm.num_units = -1;
    const long long bound = static_cast<long long>(Hq) * ((Nq + C::UNIT_ROWS - 1) / C::UNIT_ROWS + B);
    grid = bound < env.sms ? bound : env.sms;
  } else {
    prm.nqb = (Nq + C::UNIT_ROWS - 1) / C::UNIT_ROWS;
    const long long units = static_cast<long long>(B) * Hq * prm.nqb;
    if (units > 0x7fffffffLL) return FA_ERR_SHAPE;
    prm.num_units = static_cast<int>(units);
    grid = units < env.sms ? units : env.sms;
  }
  if (grid <= 0) return FA_OK;
  // The 8-bit path keeps the snake order: its K/V tiles are half the bytes,
  // its DRAM traffic is already close to the algorithmic bytes, and the
  // worker lists measured 0.4% slower on the headline workload.
  SchedTable sc;
  sc.workers = 0;
  if (soft)
    return launch_kernel(fa_fwd_kernel<D, true, SOFT_EXP_PERIOD, false>, grid, 1, C::SMEM_BYTES, stream, tq, tk, tv,
                         prm, sc);
  return launch_kernel(fa_fwd_kernel<D, true, 0, false>, grid, 1, C::SMEM_BYTES, stream, tq, tk, tv, prm, sc);
}

fa_status launch_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_descale,
                         const float* k_descale, const float* v_descale, void* o, float* lse, int B, int Hq, int Hkv,
                         int Nq, int Nk, int d, float scale, int causal, const int32_t* cu_seqlens,
                         cudaStream_t stream, const LaunchEnv& env) {
  if (d == 64)
    return launch_fp8<64>(q8, k8, vt8, q_descale, k_descale, v_descale, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal,
                          cu_seqlens, stream, env);
  return launch_fp8<128>(q8, k8, vt8, q_descale, k_descale, v_descale, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal,
                         cu_seqlens, stream, env);
}

bool fwd_schedule_for(int fp8, int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, int workers,
                      SchedTable* sc) {
  sc->workers = 0;
  if (fp8) return true;  // the 8-bit launch runs the snake order
  const int unit_rows = NQT * BLOCK_M;
  const int nqb = (Nq + unit_rows - 1) / unit_rows;
  const long long units = static_cast<long long>(B) * Hq * nqb;
  const long long grid = units < workers ? units : workers;
  sc->workers = 0;
  if (grid <= 0) return true;
  fwd_schedule(sc, 0, B, Hq, Hkv, Nq, Nk, d, 2, causal ? 1 : 0, unit_rows, nqb, units, grid);
  return true;
}

int fwd_status_and_clear() {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fa_status, sizeof(int)) != cudaSuccess) return -1;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_fa_status, &zero, sizeof(int)) != cudaSuccess) return -1;
  return v;
}

fa_status launch_exp2_soft(const float* x, float* y, int n, cudaStream_t stream) {
  const int pairs = (n + 1) / 2;
  exp2_soft_kernel<<<(pairs + 255) / 256, 256, 0, stream>>>(x, y, n);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fwd_smem_bytes(int d) {
  if (d == 64) return Cfg<64>::SMEM_BYTES;
  if (d == 128) return Cfg<128>::SMEM_BYTES;
  return 0;
}

int fwd_threads() { return NUM_THREADS; }

}  // namespace fa
