// Internal launch interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace exattn {

// Streaming multiprocessors of the current device (cached per device; 0 on
// error).  Grids of the persistent and grid-stride kernels are sized by it.
inline int device_sm_count() {
  // Launchers run outside the API lock: callers racing on a device's first
  // query store the same value.
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Raises `func`'s dynamic shared-memory limit to `bytes` once per device:
// `done` is the calling launcher's own per-device record of the value set
// (callers racing on a device's first launch set the same attribute).
inline cudaError_t smem_limit_once(const void* func, int bytes, std::atomic<int> (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_acquire) == bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev].store(bytes, std::memory_order_release);
  return e;
}

// Wait budget for every bounded pipeline wait inside the kernels.
struct DeviceGuard {
  unsigned int* status;        // device status word (OR of EXATTN_DEVICE_*_BIT)
  unsigned long long wait_ns;  // per-wait time budget
};

struct PrefillArgs {
  const CUtensorMap* tm_q;
  const CUtensorMap* tm_k;
  const CUtensorMap* tm_v;
  const CUtensorMap* tm_o;  // out, stored one 128-row tile at a time with TMA
  void* out;  // [B, Hq, Nq, d] bf16
  float* lse;
  int B, Hq, Hkv, Nq, Nk, d;
  int causal;
  float scale;
};

cudaError_t launch_prefill(const PrefillArgs& a, const DeviceGuard& g, cudaStream_t stream);
size_t prefill_smem_bytes(int d);

constexpr int kDecodeSplitTokens = 512;
constexpr int kDecodeBlockSize = 16;

struct DecodeArgs {
  const CUtensorMap* tm_k;  // cache viewed as [num_blocks * Hkv * 16 rows, d], 16-row boxes
  const CUtensorMap* tm_v;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  void* out;
  float* lse;
  float* ws_o;    // [num_seqs, Hq, max_splits, d]
  float* ws_lse;  // [num_seqs, Hq, max_splits]
  int num_seqs, Hq, Hkv, d, num_blocks, max_blocks_per_seq, max_splits;
  float scale;
};

cudaError_t launch_decode(const DecodeArgs& a, const DeviceGuard& g, cudaStream_t stream);

struct NormArgs {
  const void* x;          // [n_rows, hidden] bf16
  const void* residual;   // [n_rows, hidden] bf16
  const void* weight;     // [hidden] bf16
  void* out;              // [n_rows, hidden] bf16
  void* residual_out;     // [n_rows, hidden] bf16: x + residual
  long long n_rows;
  int hidden;             // multiple of 8, at most kNormMaxHidden
  float inv_hidden;       // 1 / hidden
  float eps;
};

constexpr int kNormMaxHidden = 16384;

cudaError_t launch_add_rms_norm(const NormArgs& a, cudaStream_t stream);

constexpr int kRopeMaxDim = 256;

struct RopeArgs {
  void* q;                    // [num_tokens, Hq, d] bf16, rotated in place
  const void* k;              // [num_tokens, Hkv, d] bf16
  const void* v;              // [num_tokens, Hkv, d] bf16
  const int32_t* seq_ids;     // [num_tokens]
  const int32_t* positions;   // [num_tokens]
  const int32_t* block_table; // [num_seqs, max_blocks_per_seq]
  void* k_cache;              // [num_blocks, Hkv, 16, d] bf16
  void* v_cache;
  unsigned int* status;       // device status word
  long long num_tokens;
  int Hq, Hkv, d, num_seqs, num_blocks, max_blocks_per_seq;
  double log2_base;
};

cudaError_t launch_rope_cache_write(const RopeArgs& a, cudaStream_t stream);

struct BwdArgs {
  // tensor maps (3-D views (d, rows, planes), 64-column boxes, 128-byte
  // swizzle) of q, dout (planes B*Hq) and k, v (planes B*Hkv), with 64-row
  // and 128-row boxes
  const CUtensorMap* tm_q64;
  const CUtensorMap* tm_do64;
  const CUtensorMap* tm_k128;
  const CUtensorMap* tm_v128;
  const CUtensorMap* tm_q128;
  const CUtensorMap* tm_do128;
  const CUtensorMap* tm_k64;
  const CUtensorMap* tm_v64;
  const CUtensorMap* tm_o128;   // out, 128-row boxes
  const CUtensorMap* tm_dq128;  // dq, 128-row boxes (TMA stores)
  const CUtensorMap* tm_ldp;    // ldp as [B*Hq][1][2 Nq] fp32, 64-pair boxes
  const void* q;     // [B, Hq, Nq, d] bf16
  const void* k;     // [B, Hkv, Nk, d] bf16
  const void* v;
  const void* out;   // forward output [B, Hq, Nq, d] bf16
  const void* dout;  // [B, Hq, Nq, d] bf16
  const float* lse;  // forward log-sum-exp [B, Hq, Nq]
  float* ldp;        // workspace: (lse * log2 e, D) pairs [B*Hq][Nq rounded up to even][2]
  float* part;       // workspace (Hq > Hkv): dK, dV partials per query head, fp32
  void* dq;          // [B, Hq, Nq, d] bf16
  void* dk;          // [B, Hkv, Nk, d] bf16
  void* dv;
  int B, Hq, Hkv, Nq, Nk, d, causal;
  float scale;
};

cudaError_t launch_bwd(const BwdArgs& a, const DeviceGuard& g, cudaStream_t stream);

}  // namespace exattn
