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
// Persistent CTAs (as many as fit on the GPU at once), each walking every
// G-th token.  Every thread copies its own 16-byte vectors of the CTA's
// next tokens into shared memory with cp.async, two tokens ahead; thread
// i < d/2 forms angle i of the next token reduced modulo 2 pi (pos *
// theta_i reaches 10^4 radians and more) and puts its cos/sin (the
// hardware fp32 approximation, within 4e-7 on the reduced angle) into
// shared memory (two buffers, so one barrier per token); each thread then
// rotates 8 pairs at a time from its two staged vectors in fp32 and rounds
// once to bf16.  The reduction needs no floating point per token:
// u_i = base^(-2i/d) / (2 pi) is held as a 64-bit fixed-point fraction of
// a turn (formed on the host, in fp64), and pos * u_i mod 2^64, an integer
// multiply, is the angle in turns, its top 32 bits read as a signed
// fraction in [-1/2, 1/2).  The error is u_i's fp64 rounding times pos
// (below 1e-10 rad for positions under 2^20) plus the final fp32 rounding,
// as with an fp64 product and reduction, and the fp64 pipe (slow on this
// GPU) is not used at all.  q is rotated in place; k is read, rotated and
// written to the cache only; v is copied to the cache.  A token whose
// sequence, position or table entry lies outside the table or the cache
// writes nothing to the cache and sets the bounds bit of the status word.
#include <cuda_bf16.h>

#include <cmath>

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

constexpr int kRopeStages = 3;  // tokens per CTA whose copies are issued (two ahead of the one in use)

// u_i = theta_i / (2 pi) per unit position, in units of 2^-64 turn, for
// i < d/2; formed on the host once per call.
struct RopeTurns {
  unsigned long long u[kRopeMaxDim / 2];
};

template <int MAXI>
constexpr size_t rope_smem_bytes() {
  return sizeof(float) * 2 * 2 * (kRopeMaxDim / 2) + sizeof(uint4) * kRopeStages * MAXI * 2 * kRopeThreads;
}

// Block-table entry of (seq, pos), or -1 when the pair lies outside the table.
__device__ __forceinline__ int table_entry(const RopeArgs& a, int seq, int pos) {
  if (seq < 0 || seq >= a.num_seqs || pos < 0 || pos / 16 >= a.max_blocks_per_seq) return -1;
  return a.block_table[static_cast<long long>(seq) * a.max_blocks_per_seq + pos / 16];
}

// MAXI: work items per thread per token (q and k items are 8 pairs from
// two 16-byte vectors, v items one 16-byte copy); which items a thread owns
// and where they sit within a token's rows is the same for every token and
// worked out once.  Each thread copies its own vectors of the CTA's next
// tokens into its own shared-memory slots with cp.async, kRopeStages - 1
// tokens ahead of the one it rotates, so the loads stay in flight without
// holding registers and need no barrier (a thread reads back only what it
// copied).  The token metadata runs ahead too: position and sequence two
// tokens ahead, the block-table entry one token ahead, so no dependent load
// sits inside an iteration; and the cos/sin of the next token's angles are
// formed right after the barrier that publishes the current token's, into
// the other buffer, so that barrier does not wait for them.
template <int MAXI>
__global__ void __launch_bounds__(kRopeThreads) rope_cache_kernel(const RopeArgs a, const RopeTurns turns) {
  extern __shared__ __align__(16) uint8_t rope_smem[];
  float(*const cs)[2][kRopeMaxDim / 2] = reinterpret_cast<float(*)[2][kRopeMaxDim / 2]>(rope_smem);
  uint4(*const stage)[MAXI][2][kRopeThreads] = reinterpret_cast<uint4(*)[MAXI][2][kRopeThreads]>(
      rope_smem + sizeof(float) * 2 * 2 * (kRopeMaxDim / 2));
  const int tid = threadIdx.x;
  const int d = a.d, half = d / 2, vec_half = half / 8, vec_d = d / 8;
  // angle tid (if < half; half <= kRopeThreads)
  const unsigned long long u_turn = tid < half ? turns.u[tid] : 0ull;
  uint4* q = static_cast<uint4*>(a.q);
  const uint4* k = static_cast<const uint4*>(a.k);
  const uint4* v = static_cast<const uint4*>(a.v);
  uint4* kc = static_cast<uint4*>(a.k_cache);
  uint4* vc = static_cast<uint4*>(a.v_cache);
  const long long G = gridDim.x, T = a.num_tokens;
  const size_t q_tok = static_cast<size_t>(a.Hq) * vec_d;    // 16-byte vectors per token of q
  const size_t kv_tok = static_cast<size_t>(a.Hkv) * vec_d;  // ... of k or v

  // Items: q heads x vec_half, then k heads x vec_half, then v heads x vec_d.
  // kind 0 q, 1 k, 2 v, 3 none; off = vector within the token's rows; coff =
  // vector within the token's cache rows (k, v); jv = first pair / 8 (q, k).
  const int n_q = a.Hq * vec_half, n_k = a.Hkv * vec_half, n_all = n_q + n_k + a.Hkv * vec_d;
  int kind[MAXI], off[MAXI], coff[MAXI], jv[MAXI];
#pragma unroll
  for (int i = 0; i < MAXI; ++i) {
    const int w = tid + i * kRopeThreads;
    kind[i] = 3;
    off[i] = coff[i] = jv[i] = 0;
    if (w < n_q) {
      kind[i] = 0;
      jv[i] = w % vec_half;
      off[i] = (w / vec_half) * vec_d + jv[i];
    } else if (w < n_q + n_k) {
      const int item = w - n_q;
      kind[i] = 1;
      jv[i] = item % vec_half;
      off[i] = (item / vec_half) * vec_d + jv[i];
      coff[i] = (item / vec_half) * 16 * vec_d + jv[i];
    } else if (w < n_all) {
      const int item = w - n_q - n_k;
      kind[i] = 2;
      off[i] = item;
      coff[i] = (item / vec_d) * 16 * vec_d + item % vec_d;
    }
  }

  // This thread's copies of token t into stage st; one commit group per
  // call (empty past the last token), so the group count stays uniform.
  auto issue = [&](long long t, int st) {
    if (t < T) {
      const uint4* qs = q + static_cast<size_t>(t) * q_tok;
      const uint4* ks = k + static_cast<size_t>(t) * kv_tok;
      const uint4* vs = v + static_cast<size_t>(t) * kv_tok;
#pragma unroll
      for (int i = 0; i < MAXI; ++i) {
        const uint32_t lo = smem_u32(&stage[st][i][0][tid]), hi = smem_u32(&stage[st][i][1][tid]);
        if (kind[i] == 0) {
          cp_async16(lo, qs + off[i], true);
          cp_async16(hi, qs + off[i] + vec_half, true);
        } else if (kind[i] == 1) {
          cp_async16(lo, ks + off[i], true);
          cp_async16(hi, ks + off[i] + vec_half, true);
        } else if (kind[i] == 2) {
          cp_async16(lo, vs + off[i], true);
        }
      }
    }
    cp_async_commit();
  };
  // cos/sin of angle tid of position pos into buffer buf.  pos * u mod 2^64
  // is the angle in 2^-64 turns; its top 32 bits as a signed fraction of a
  // turn times 2 pi give it in [-pi, pi), where the hardware sin/cos
  // approximation is within 4e-7 absolute.
  auto angles = [&](int pos, int buf) {
    if (tid < half) {
      const unsigned long long turn = static_cast<unsigned long long>(static_cast<long long>(pos)) * u_turn;
      const int top = static_cast<int>(static_cast<unsigned int>(turn >> 32));
      const float r = static_cast<float>(top) * 1.46291807926715968e-9f;  // 2 pi / 2^32
      float sn, cn;
      __sincosf(r, &sn, &cn);
      cs[buf][0][tid] = cn;
      cs[buf][1][tid] = sn;
    }
  };

  long long t = blockIdx.x;
#pragma unroll
  for (int st = 0; st < kRopeStages - 1; ++st) issue(t + st * G, st);
  int pos0 = t < T ? a.positions[t] : 0, seq0 = t < T ? a.seq_ids[t] : -1;
  int pos1 = t + G < T ? a.positions[t + G] : 0, seq1 = t + G < T ? a.seq_ids[t + G] : -1;
  int blk0 = table_entry(a, seq0, pos0);
  angles(pos0, 0);
  for (int n = 0; t < T; ++n, t += G) {
    issue(t + (kRopeStages - 1) * G, (n + kRopeStages - 1) % kRopeStages);
    const int blk1 = table_entry(a, seq1, pos1);  // used in the next iteration
    const long long t2 = t + 2 * G;
    const int pos2 = t2 < T ? a.positions[t2] : 0, seq2 = t2 < T ? a.seq_ids[t2] : -1;
    const long long slot = (blk0 >= 0 && blk0 < a.num_blocks) ? static_cast<long long>(blk0) * 16 + pos0 % 16 : -1;
    if (slot < 0 && tid == 0) atomicOr(a.status, 2u);  // EXATTN_DEVICE_BOUNDS_BIT
    cp_async_wait<kRopeStages - 1>();  // this thread's copies of token t have landed
    // Publishes cs[n & 1]; every read of cs[(n + 1) & 1] (token t - G)
    // happened before it, so the next token's angles may go there now.
    __syncthreads();
    if (t + G < T) angles(pos1, (n + 1) & 1);

    float(*const csp)[kRopeMaxDim / 2] = cs[n & 1];
    const int st = n % kRopeStages;
    uint4* qd = q + static_cast<size_t>(t) * q_tok;
    const size_t cache_row =
        slot >= 0 ? (static_cast<size_t>(slot / 16) * a.Hkv * 16 + slot % 16) * vec_d : 0;
#pragma unroll
    for (int i = 0; i < MAXI; ++i) {
      uint4 lo = stage[st][i][0][tid], hi = stage[st][i][1][tid];
      if (kind[i] == 0) {
        rotate8(lo, hi, &csp[0][8 * jv[i]], &csp[1][8 * jv[i]]);
        qd[off[i]] = lo;
        qd[off[i] + vec_half] = hi;
      } else if (kind[i] == 1) {
        rotate8(lo, hi, &csp[0][8 * jv[i]], &csp[1][8 * jv[i]]);
        if (slot >= 0) {
          kc[cache_row + coff[i]] = lo;
          kc[cache_row + coff[i] + vec_half] = hi;
        }
      } else if (kind[i] == 2 && slot >= 0) {
        vc[cache_row + coff[i]] = lo;
      }
    }
    pos0 = pos1;
    blk0 = blk1;
    pos1 = pos2;
    seq1 = seq2;
  }
  cp_async_wait<0>();  // the groups still open are empty; none stays behind the CTA
}

template <int MAXI>
cudaError_t launch_maxi(const RopeArgs& a, const RopeTurns& turns, int sms, cudaStream_t stream) {
  constexpr size_t smem = rope_smem_bytes<MAXI>();
  // CTAs per SM, per device, set up on the device's first call (callers
  // racing on it set the same attribute and store the same value)
  static std::atomic<int> resident[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int r = resident[dev].load(std::memory_order_acquire);
  if (r == 0) {
    e = cudaFuncSetAttribute(rope_cache_kernel<MAXI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, rope_cache_kernel<MAXI>, kRopeThreads, smem);
    if (e != cudaSuccess) return e;
    if (r < 1) return cudaErrorInvalidConfiguration;
    resident[dev].store(r, std::memory_order_release);
  }
  const long long cap = static_cast<long long>(sms) * r;
  const int grid = static_cast<int>(a.num_tokens < cap ? a.num_tokens : cap);
  rope_cache_kernel<MAXI><<<grid, kRopeThreads, smem, stream>>>(a, turns);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rope_cache_write(const RopeArgs& a, cudaStream_t stream) {
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  if (a.d < 16 || a.d > kRopeMaxDim || a.d % 16 != 0) return cudaErrorInvalidValue;
  // theta_i / (2 pi) * 2^64 = base^(-2i/d) * 2^64 / (2 pi), below 2^62, rounded to an integer
  RopeTurns turns{};
  for (int i = 0; i < a.d / 2; ++i)
    turns.u[i] = static_cast<unsigned long long>(
        std::nearbyint(std::exp2(-(2.0 * i / a.d) * a.log2_base) * (18446744073709551616.0 / 6.283185307179586476925)));
  const long long items = static_cast<long long>(a.Hq) * (a.d / 16) +
                          static_cast<long long>(a.Hkv) * (a.d / 16) + static_cast<long long>(a.Hkv) * (a.d / 8);
  const long long per_thread = (items + kRopeThreads - 1) / kRopeThreads;
  if (per_thread <= 1) return launch_maxi<1>(a, turns, sms, stream);
  if (per_thread <= 2) return launch_maxi<2>(a, turns, sms, stream);
  if (per_thread <= 4) return launch_maxi<4>(a, turns, sms, stream);
  if (per_thread <= 8) return launch_maxi<8>(a, turns, sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace exattn
