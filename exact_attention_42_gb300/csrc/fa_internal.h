// Host-side declarations shared by the translation units of libfa.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "fa.h"

namespace fa {

constexpr int kMaxDevicesDecode = 64;                      // devices with per-device launch state
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;  // bound on every kernel wait: 2 s

// Fault-injection modes of fa_debug_fault_injection: which kernel's ring
// producer withholds its first copy.
constexpr int kFaultNone = 0;
constexpr int kFaultFwd = 1;     // fa_fwd_kernel's K/V producer
constexpr int kFaultDecode = 2;  // decode_kernel's K/V producer
constexpr int kFaultBwdDq = 3;   // bwd_dq_kernel's K/V producer
constexpr int kFaultBwdDkdv = 4; // bwd_dkdv_kernel's Q/dO producer
constexpr int kFaultQuant = 5;   // quant_fused_kernel's first bulk copy in every CTA
constexpr int kFaultModes = 6;

// Launch configuration with programmatic stream serialization: the kernel
// may start before the previous kernel in `stream` has finished, runs its
// shared-memory and TMEM set-up meanwhile, and waits for that kernel
// (griddepcontrol.wait) before it touches global memory.  cluster_x > 1
// launches clusters of that many CTAs.  cfg points into this object, so it
// is used in place: PdlLaunch L(...); cudaLaunchKernelEx(&L.cfg, ...).
struct PdlLaunch {
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[2];
  PdlLaunch(dim3 grid, unsigned threads, size_t smem, cudaStream_t stream, unsigned cluster_x = 1) {
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cluster_x > 1 ? 2 : 1;
  }
  PdlLaunch(const PdlLaunch&) = delete;
  PdlLaunch& operator=(const PdlLaunch&) = delete;
};

// Per-call launch settings resolved by the entry points (fa_api.cu).
struct LaunchEnv {
  int device = 0;
  int sms = 0;                          // streaming multiprocessors of the device
  unsigned long long wait_limit_ns = 0;  // bound on every mbarrier wait
  int fault_mode = 0;                   // test hook, see fa_debug_fault_injection
  int soft_exp = 0;                     // test hook, see fa_debug_soft_exp
  int fwd_pair = 0;                     // test hook, see fa_debug_fwd_pair
};

// Unit lists of a persistent launch, one per worker (CTA, or CTA pair),
// handed to the kernel by value as a __grid_constant__ parameter, so they need
// no device memory.  Worker w runs units unit[start[w] .. start[w+1]) in that
// order.  workers == 0 means no table: the kernel deals units in its static
// snake order instead (packed sequences, whose lengths the host does not
// know, and problems larger than the table).
constexpr int kSchedMaxWorkers = 160;
constexpr int kSchedCap = 4096;
struct SchedTable {
  int workers;
  uint16_t start[kSchedMaxWorkers + 1];
  uint16_t unit[kSchedCap];
};

// How the schedule builder sees unit u: its predicted cost (K/V or Q/dO tile
// steps plus a fixed per-unit overhead, in steps) and the group of heads whose
// tiles it streams.  Groups are sized so that the tiles of one group stay
// resident in L2 (kSchedGroupBytes), and are visited one after another.
struct SchedUnit {
  float cost;
  int group;
};
constexpr double kSchedGroupBytes = 32.0 * 1024 * 1024;
// Heads per group when one head streams `bytes_per_head` bytes.
int sched_group_heads(double bytes_per_head);
// Fills *out for `units` units over `workers` workers: units are taken group
// by group, longest first within a group, and each goes to the worker the
// costs predict to be free first (list scheduling, LPT order within groups).
// Results are cached per process under `key` (the launch's shape).  Returns
// false, with out->workers = 0, when the problem does not fit the table.
bool build_schedule(const long long (&key)[12], int workers, int units, void (*describe)(const void*, int, SchedUnit*),
                    const void* ctx, SchedTable* out);

// The table a dense single-CTA forward launch over `workers` workers uses
// (fa_fwd.cu; for fa_debug_schedule).
bool fwd_schedule_for(int fp8, int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, int workers,
                      SchedTable* sc);

// The same for the backward dQ (kv = 0) or dK/dV (kv = 1) kernel (fa_bwd.cu).
bool bwd_schedule_for(int kv, int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, int workers,
                      SchedTable* sc);

// FA_OK if the current device is supported (sm_103), FA_ERR_UNSUPPORTED
// otherwise, FA_ERR_CUDA if it cannot be queried (fa_api.cu).
fa_status check_device();

// Forward kernel (fa_fwd.cu); dispatches to the split-KV path itself.
fa_status launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                     int Nq, int Nk, int d, float scale, int causal, const int32_t* cu_seqlens, cudaStream_t stream,
                     const LaunchEnv& env);
// 8-bit forward (fa_fwd.cu, d = 64 or 128, dense or packed): e4m3 Q, K and
// V^T with per-(batch, head) descales (per head when packed).
fa_status launch_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_descale,
                         const float* k_descale, const float* v_descale, void* o, float* lse, int B, int Hq, int Hkv,
                         int Nq, int Nk, int d, float scale, int causal, const int32_t* cu_seqlens,
                         cudaStream_t stream, const LaunchEnv& env);
int fwd_status_and_clear();  // -1 if the status word cannot be read
// e4m3 codes and per-(batch, head) descales of a bf16 tensor (fa_quant.cu).
fa_status launch_fp8_quantize(const void* x, void* x8, float* descale, int B, int H, int N, int d, int transpose,
                              const int8_t* signs, cudaStream_t stream, const LaunchEnv& env);
int quant_status_and_clear();  // -1 if the status word cannot be read
fa_status launch_exp2_soft(const float* x, float* y, int n, cudaStream_t stream);
int fwd_smem_bytes(int d);
int fwd_threads();

// Tensor map of a [heads, rows, d] bf16 tensor read in boxes of 64 columns x
// box_rows rows with the 128-byte swizzle; false if the CUDA driver rejects it.
bool encode_bf16_rows_map(CUtensorMap* map, const void* base, int d, long long rows, long long heads, int box_rows);

// Split-KV path (fa_decode.cu) for dense problems with (Hq / Hkv) * Nq <= 16.
bool decode_supported(int B, int Hq, int Hkv, int Nq, int Nk, int d, const int32_t* cu_seqlens);
fa_status launch_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int Nq, int Nk, int d, float scale, int causal, cudaStream_t stream, int sms,
                        unsigned long long wait_limit_ns, int fault_mode);
int decode_status_and_clear();  // -1 if the status word cannot be read
int decode_smem_bytes(int d);

// Backward pass (fa_bwd.cu), dense or packed layout.
fa_status launch_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                     void* dq, void* dk, void* dv, float* delta, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                     float scale, int causal, const int32_t* cu_seqlens, cudaStream_t stream, int sms,
                     unsigned long long wait_limit_ns, int fault_mode);
int bwd_status_and_clear();  // -1 if the status word cannot be read
int bwd_smem_bytes(int d);

}  // namespace fa
