// Rotary position embedding + paged KV-cache write for sm_103a.
//
// For every new token t (of sequence seq_ids[t], at position positions[t]):
// rotate each query and key head vector by the token's position, then store
// the rotated key and the value into the token's slot of the block-paged
// cache, in one pass ("Inference Engineering VII.07: Kernel and Operator
// Fusion" page, section 2, "rope + cache write: RoPE then KV store";
// "Fused Kernel Compiler" page, table of fusion patterns, "RoPE embedding:
// sin, cos, rotate").  Pairs (i, i + d/2) turn by theta_i = pos *
// base^(-2i/d):
//   y_i = x_i cos - x_(i+d/2) sin,   y_(i+d/2) = x_(i+d/2) cos + x_i sin.
// The slot is pos % 16 of physical block block_table[seq][pos / 16]
// ("Optimizing LLM Inference ..." page, section Paged Attention and Dynamic
// KV Cache Management); cache [num_blocks, Hkv, 16, d].
//
// One CTA per token (grid-stride; the d/2 frequencies are computed once per
// CTA in fp64): every thread first loads its vectors of the token, then the
// d/2 angles are formed and reduced
// modulo 2 pi in fp64 (pos * inv_freq reaches 10^4 radians and more), then
// cos/sin of the reduced angle in fp32 go to shared memory; each thread then
// rotates 8 pairs at a time from two 16-byte vectors in fp32 and rounds once
// to bf16.  q is rotated in place; k is read, rotated and written to the
// cache only; v is copied to the cache.  A token whose sequence, position
// or table entry lies outside the table or the cache writes nothing to the
// cache and sets the bounds bit of the status word.
#include <cuda_bf16.h>

#include "launch.h"
#include "ptx.cuh"

namespace exattn {
namespace {

constexpr int kRopeThreads = 256;

// Rotates the 8 pairs (lo[e], hi[e]) by angles with cosines c[e], sines s[e].
__device__ __forceinline__ void rotate8(uint4& lo, uint4& hi, const float* c, const float* s) {
  float a[8], b[8], ya[8], yb[8];
  unpack_bf16x8(lo, a);
  unpack_bf16x8(hi, b);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    ya[e] = fmaf(a[e], c[e], -b[e] * s[e]);
    yb[e] = fmaf(b[e], c[e], a[e] * s[e]);
  }
  lo = pack_bf16x8(ya);
  hi = pack_bf16x8(yb);
}

// MAXI: work items per thread per token (q and k items are 8 pairs, v items
// one 16-byte copy).  Each thread first issues the loads of all its items,
// then the token's angles are formed, so the loads are in flight meanwhile.
// (Two tokens per CTA step measured slower: fewer CTAs on a decode step and
// more registers per thread.)
template <int MAXI>
__global__ void __launch_bounds__(kRopeThreads) rope_cache_kernel(const RopeArgs a) {
  __shared__ double inv_freq[kRopeMaxDim / 2];  // base^(-2i/d), the same for every token
  __shared__ float cs[2][kRopeMaxDim / 2];        // cos, sin of this token's angles
  const int d = a.d, half = d / 2, vec_half = half / 8, vec_d = d / 8;
  for (int i = threadIdx.x; i < half; i += kRopeThreads) inv_freq[i] = exp2(-(2.0 * i / d) * a.log2_base);
  __syncthreads();
  uint4* q = static_cast<uint4*>(a.q);
  const uint4* k = static_cast<const uint4*>(a.k);
  const uint4* v = static_cast<const uint4*>(a.v);
  uint4* kc = static_cast<uint4*>(a.k_cache);
  uint4* vc = static_cast<uint4*>(a.v_cache);
  // q: Hq heads x vec_half items; k: Hkv heads x vec_half; v: Hkv x vec_d copies
  const int n_q = a.Hq * vec_half, n_k = a.Hkv * vec_half, n_all = n_q + n_k + a.Hkv * vec_d;
  for (long long t = blockIdx.x; t < a.num_tokens; t += gridDim.x) {
    uint4 lo[MAXI], hi[MAXI];
#pragma unroll
    for (int i = 0; i < MAXI; ++i) {
      const int w = threadIdx.x + i * kRopeThreads;
      if (w < n_q) {
        const size_t row = (static_cast<size_t>(t) * a.Hq + w / vec_half) * vec_d + w % vec_half;
        lo[i] = q[row];
        hi[i] = q[row + vec_half];
      } else if (w < n_q + n_k) {
        const int item = w - n_q;
        const size_t row = (static_cast<size_t>(t) * a.Hkv + item / vec_half) * vec_d + item % vec_half;
        lo[i] = k[row];
        hi[i] = k[row + vec_half];
      } else if (w < n_all) {
        const int item = w - n_q - n_k;
        lo[i] = v[(static_cast<size_t>(t) * a.Hkv + item / vec_d) * vec_d + item % vec_d];
      }
    }
    const int pos = a.positions[t];
    const int seq = a.seq_ids[t];
    long long slot = -1;  // block * 16 + offset
    if (seq >= 0 && seq < a.num_seqs && pos >= 0 && pos / 16 < a.max_blocks_per_seq) {
      const int blk = a.block_table[static_cast<long long>(seq) * a.max_blocks_per_seq + pos / 16];
      if (blk >= 0 && blk < a.num_blocks) slot = static_cast<long long>(blk) * 16 + pos % 16;
    }
    if (slot < 0 && threadIdx.x == 0) atomicOr(a.status, 2u);  // EXATTN_DEVICE_BOUNDS_BIT
    for (int i = threadIdx.x; i < half; i += kRopeThreads) {
      const double ang = static_cast<double>(pos) * inv_freq[i];
      const double r = ang - 6.283185307179586476925 * rint(ang * 0.159154943091895335769);
      float sn, cn;
      sincosf(static_cast<float>(r), &sn, &cn);
      cs[0][i] = cn;
      cs[1][i] = sn;
    }
    __syncthreads();
    const size_t cache_row =
        slot >= 0 ? (static_cast<size_t>(slot / 16) * a.Hkv * 16 + slot % 16) * vec_d : 0;
#pragma unroll
    for (int i = 0; i < MAXI; ++i) {
      const int w = threadIdx.x + i * kRopeThreads;
      if (w < n_q) {
        const int j = w % vec_half;
        rotate8(lo[i], hi[i], &cs[0][8 * j], &cs[1][8 * j]);
        const size_t row = (static_cast<size_t>(t) * a.Hq + w / vec_half) * vec_d + j;
        q[row] = lo[i];
        q[row + vec_half] = hi[i];
      } else if (w < n_q + n_k) {
        const int item = w - n_q, j = item % vec_half;
        rotate8(lo[i], hi[i], &cs[0][8 * j], &cs[1][8 * j]);
        if (slot >= 0) {
          const size_t dst = cache_row + static_cast<size_t>(item / vec_half) * 16 * vec_d + j;
          kc[dst] = lo[i];
          kc[dst + vec_half] = hi[i];
        }
      } else if (w < n_all && slot >= 0) {
        const int item = w - n_q - n_k;
        vc[cache_row + static_cast<size_t>(item / vec_d) * 16 * vec_d + item % vec_d] = lo[i];
      }
    }
    __syncthreads();  // cs is refilled for the next token
  }
}

}  // namespace

cudaError_t launch_rope_cache_write(const RopeArgs& a, cudaStream_t stream) {
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const long long cap = static_cast<long long>(sms) * 8;
  const int grid = static_cast<int>(a.num_tokens < cap ? a.num_tokens : cap);
  const long long items = static_cast<long long>(a.Hq) * (a.d / 16) +
                          static_cast<long long>(a.Hkv) * (a.d / 16) + static_cast<long long>(a.Hkv) * (a.d / 8);
  const long long per_thread = (items + kRopeThreads - 1) / kRopeThreads;
  if (per_thread <= 1) rope_cache_kernel<1><<<grid, kRopeThreads, 0, stream>>>(a);
  else if (per_thread <= 2) rope_cache_kernel<2><<<grid, kRopeThreads, 0, stream>>>(a);
  else if (per_thread <= 4) rope_cache_kernel<4><<<grid, kRopeThreads, 0, stream>>>(a);
  else if (per_thread <= 8) rope_cache_kernel<8><<<grid, kRopeThreads, 0, stream>>>(a);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace exattn
