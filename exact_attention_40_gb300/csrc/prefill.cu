// Prefill attention kernel for sm_103a.
//
// One CTA computes one 128-row query tile of one (batch, query head):
//   O = softmax(scale * Q K^T + mask) V,  lse = log sum exp(scale * Q K^T)
// streaming the keys/values of the mapped KV head in 128-row tiles, with
// an online softmax so the score tile S and probability tile P exist only
// in tensor memory / shared memory ("Fused Kernel Compiler" page,
// subsection FlashAttention Integration, items 1-4).
//
// Warp roles (192 threads):
//   warps 0-3  softmax warpgroup: thread r owns query row r of the tile,
//              which is TMEM lane r.  Reads S from TMEM, applies the mask,
//              keeps the running max m and sum l, writes P (bf16) to shared
//              memory, rescales O in TMEM when m grows by more than
//              kRescaleThreshold (log2 units), and runs the epilogue.
//   warp 4     TMA producer: Q once, then K_j / V_j tiles into two rings.
//   warp 5     tcgen05 issuer (one thread): S_j = Q K_j^T into one of two
//              TMEM S buffers, then O += P_{j-1} V_{j-1}; also owns the TMEM
//              allocation.
//
// TMEM (512 columns): S0 [0,128), S1 [128,256), O [256, 256+d).
// Shared memory: every operand tile is stored as 128-row x 64-column bf16
// sub-tiles (16 KB, 128-byte swizzle) exactly as TMA writes them; the MMA
// descriptors read them in place (K-major for Q, K and P; MN-major for V).
#include <cuda_bf16.h>

#include "launch.h"
#include "ptx.cuh"

namespace exattn {
namespace {

constexpr int kBM = 128;                  // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;                  // keys per tile
constexpr int kThreads = 192;
constexpr int kWarpLoad = 4;
constexpr int kWarpMma = 5;
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;          // column of the O accumulator
constexpr float kRescaleThreshold = 8.0f; // log2 units: p may reach 2^8 before O is rescaled
constexpr uint32_t kSubTileBytes = 128 * 64 * 2;

template <int D>
struct alignas(1024) PrefillSmem {
  uint8_t q[D / 64][kSubTileBytes];            // Q tile; reused as O staging
  uint8_t k[kKStages][D / 64][kSubTileBytes];  // K ring
  uint8_t v[kVStages][D / 64][kSubTileBytes];  // V ring
  uint8_t p[kBN / 64][kSubTileBytes];          // P tile (bf16)
  uint64_t q_full;
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, o_done, mma_fin;
  uint32_t tmem_base;
  uint32_t abort_flag;
};

struct KernelParams {
  float* lse;
  unsigned int* status;
  unsigned long long wait_ns;
  int Hq, Hkv, Nq, Nk, group, n_qtiles, causal;
  float scale_log2;  // scale * log2(e)
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              const KernelParams& p, uint32_t* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  volatile uint32_t* ab = abort_flag;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*ab) return false;
    if (globaltimer_ns() - t0 > p.wait_ns) {
      atomicOr(p.status, 1u);  // EXATTN_DEVICE_TIMEOUT_BIT
      *ab = 1u;
      return false;
    }
  }
}

__device__ __forceinline__ void named_bar_softmax() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const KernelParams p) {
  extern __shared__ uint8_t smem_raw[];
  PrefillSmem<D>& sm = *reinterpret_cast<PrefillSmem<D>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work item: late (heavier under the causal mask) query tiles launch first.
  const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x);
  const int hq = blockIdx.y;
  const int b = blockIdx.z;
  const int hkv = hq / p.group;
  const int m0 = qt * kBM;
  const int zq = b * p.Hq + hq;
  const int zk = b * p.Hkv + hkv;

  // Key tiles this query tile needs, and how many of them need no mask.
  const long long shift = static_cast<long long>(p.Nk) - p.Nq;  // bottom-right alignment
  int n_kv = (p.Nk + kBN - 1) / kBN;
  int n_full = p.Nk / kBN;
  if (p.causal) {
    const long long last = static_cast<long long>(m0) + kBM - 1 + shift;  // last key of last row
    const int lim = last < 0 ? 0 : static_cast<int>(last / kBN) + 1;
    n_kv = min(n_kv, lim);
    const long long first = static_cast<long long>(m0) + shift + 1;  // keys visible to row m0
    const int full_c = first <= 0 ? 0 : static_cast<int>(first / kBN);
    n_full = min(n_full, full_c);
  }

  if (warp == kWarpLoad && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
    mbar_init(&sm.q_full, 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.s_full[s], 1);
      mbar_init(&sm.s_free[s], 128);
    }
    mbar_init(&sm.p_full, 128);
    mbar_init(&sm.o_done, 1);
    mbar_init(&sm.mma_fin, 1);
    sm.abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    __syncwarp();
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sm.tmem_base;

  int issued_k[kKStages] = {0, 0};
  int issued_v[kVStages] = {0, 0};
  bool issued_q = false;
  bool mma_issued = false;

  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_kv > 0) {
      const uint64_t keep = l2_policy_evict_last();  // K/V tiles are re-read by other CTAs
      mbar_arrive_expect_tx(&sm.q_full, D * kBM * 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tma_load_3d(sm.q[c], &tm_q, &sm.q_full, c * 64, m0, zq);
      issued_q = true;
      for (int j = 0; j < n_kv; ++j) {
        const int sk = j % kKStages;
        if (j >= kKStages && !wait_or_abort(&sm.k_empty[sk], ((j / kKStages) - 1) & 1, p, &sm.abort_flag))
          break;
        mbar_arrive_expect_tx(&sm.k_full[sk], D * kBN * 2);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d_hint(sm.k[sk][c], &tm_k, &sm.k_full[sk], c * 64, j * kBN, zk, keep);
        issued_k[sk] = j / kKStages + 1;
        const int sv = j % kVStages;
        if (j >= kVStages && !wait_or_abort(&sm.v_empty[sv], ((j / kVStages) - 1) & 1, p, &sm.abort_flag))
          break;
        mbar_arrive_expect_tx(&sm.v_full[sv], D * kBN * 2);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d_hint(sm.v[sv][c], &tm_v, &sm.v_full[sv], c * 64, j * kBN, zk, keep);
        issued_v[sv] = j / kVStages + 1;
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_kv > 0) {
      constexpr uint32_t id_qk = idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t id_pv = idesc_bf16_f32(kBM, D, false, true);
      bool ok = wait_or_abort(&sm.q_full, 0, p, &sm.abort_flag);
      tc_fence_after_sync();
      for (int j = 0; ok && j <= n_kv; ++j) {
        if (j < n_kv) {
          const int sk = j % kKStages;
          if (!wait_or_abort(&sm.k_full[sk], (j / kKStages) & 1, p, &sm.abort_flag)) break;
          if (j >= 2 && !wait_or_abort(&sm.s_free[j & 1], ((j >> 1) - 1) & 1, p, &sm.abort_flag)) break;
          tc_fence_after_sync();
          const uint32_t d_s = tmem + static_cast<uint32_t>(j & 1) * kBN;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t a = smem_desc(smem_u32(sm.q[kk / 4]) + (kk % 4) * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(smem_u32(sm.k[sk][kk / 4]) + (kk % 4) * 32, 16, 1024, kSwizzle128B);
            umma_bf16_ss(d_s, a, bd, id_qk, kk > 0 ? 1u : 0u);
          }
          mma_issued = true;
          umma_commit(&sm.s_full[j & 1]);
          umma_commit(&sm.k_empty[sk]);
        }
        if (j >= 1) {
          const int jj = j - 1;
          const int sv = jj % kVStages;
          if (!wait_or_abort(&sm.v_full[sv], (jj / kVStages) & 1, p, &sm.abort_flag)) break;
          if (!wait_or_abort(&sm.p_full, jj & 1, p, &sm.abort_flag)) break;
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            const uint64_t a = smem_desc(smem_u32(sm.p[kk / 4]) + (kk % 4) * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(smem_u32(sm.v[sv][0]) + kk * 2048, kSubTileBytes, 1024, kSwizzle128B);
            umma_bf16_ss(tmem + kTmemO, a, bd, id_pv, (jj > 0 || kk > 0) ? 1u : 0u);
          }
          mma_issued = true;
          umma_commit(&sm.v_empty[sv]);
          umma_commit(&sm.o_done);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroup
    const int r = warp * 32 + lane;  // row within the tile == TMEM lane
    const int row = m0 + r;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const long long vis_last = static_cast<long long>(row) + shift;  // causal: keys <= vis_last
    float m_ref = -INFINITY;  // reference max, log2 units
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!__all_sync(0xffffffffu, wait_or_abort(&sm.s_full[j & 1], (j >> 1) & 1, p, &sm.abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      uint32_t sr[kBN];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c)
        tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(j & 1) * kBN + c * 32,
                           *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
      tmem_ld_wait();
      tc_fence_before_sync();
      mbar_arrive(&sm.s_free[j & 1]);

      float s[kBN];
#pragma unroll
      for (int c = 0; c < kBN; ++c) s[c] = __uint_as_float(sr[c]);
      if (j >= n_full) {
        const long long key0 = static_cast<long long>(j) * kBN;
        long long lim = static_cast<long long>(p.Nk) - key0;  // keys >= Nk do not exist
        if (p.causal) lim = min(lim, vis_last - key0 + 1);
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (c >= lim) s[c] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < kBN; ++c) mx = fmaxf(mx, s[c]);
      mx *= p.scale_log2;
      float alpha = 1.f;
      bool rescale = false;
      if (mx > m_ref + kRescaleThreshold) {
        alpha = ex2_approx(m_ref - mx);  // 0 when m_ref is -inf
        m_ref = mx;
        rescale = true;
      }
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      float sum = 0.f;
      uint32_t pk[kBN / 2];
#pragma unroll
      for (int c = 0; c < kBN / 2; ++c) {
        const float p0 = ex2_approx(fmaf(s[2 * c], p.scale_log2, -m_use));
        const float p1 = ex2_approx(fmaf(s[2 * c + 1], p.scale_log2, -m_use));
        sum += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + sum;

      // P buffer and O are owned by the previous P*V until it completes.
      if (j >= 1 && !__all_sync(0xffffffffu, wait_or_abort(&sm.o_done, (j - 1) & 1, p, &sm.abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      // tcgen05.ld/st are warp-collective: the whole warp rescales if any
      // of its rows needs it (alpha is 1 for the others).
      if (__any_sync(0xffffffffu, rescale) && j >= 1) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(t_lane + kTmemO + c * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st_32x32b_x32(t_lane + kTmemO + c * 32, o);
        }
        tmem_st_wait();
      }
      // P row r -> two K-major swizzled sub-tiles (16-byte chunk c of a
      // 128-byte row lands at chunk c ^ (row & 7)).
#pragma unroll
      for (int ch = 0; ch < kBN / 8; ++ch) {
        const uint32_t base = smem_u32(sm.p[ch / 8]) + r * 128;
        const uint32_t addr = base + (((ch % 8) ^ (r & 7)) << 4);
        st_shared_v4(addr, pk[ch * 4 + 0], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(&sm.p_full);
    }

    // ------------------------------------------------------------ epilogue
    if (ok && n_kv > 0)
      ok = __all_sync(0xffffffffu, wait_or_abort(&sm.o_done, (n_kv - 1) & 1, p, &sm.abort_flag));
    tc_fence_after_sync();
    const bool have = ok && n_kv > 0;  // warp-uniform
    const bool row_has_keys = have && l > 0.f;
    const float inv_l = row_has_keys ? 1.f / l : 0.f;
    if (p.lse != nullptr && row < p.Nq) {
      const float lse = row_has_keys ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      p.lse[static_cast<size_t>(zq) * p.Nq + row] = lse;
    }
    // O row -> bf16 -> swizzled staging in the (now idle) Q buffer.
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      if (have) {
        tmem_ld_32x32b_x32(t_lane + kTmemO + c * 32, o);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
      uint32_t w[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
      const uint32_t base = smem_u32(sm.q[c / 2]) + r * 128;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int ch = (c % 2) * 4 + i;
        st_shared_v4(base + ((ch ^ (r & 7)) << 4), w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      }
    }
    fence_proxy_async_smem();
    named_bar_softmax();
    if (r == 0) {
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tma_store_3d(&tm_o, sm.q[c], c * 64, m0, zq);
      bulk_commit_group();
      bulk_wait_group_read0();
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  const bool aborted = *reinterpret_cast<volatile uint32_t*>(&sm.abort_flag) != 0u;
  if (aborted) {
    // Drain what is still in flight before the CTA's memory goes away.
    if (warp == kWarpLoad && lane == 0) {
      if (issued_q) mbar_wait(&sm.q_full, 0, p.wait_ns);
      for (int s = 0; s < kKStages; ++s)
        if (issued_k[s] > 0) mbar_wait(&sm.k_full[s], (issued_k[s] - 1) & 1, p.wait_ns);
      for (int s = 0; s < kVStages; ++s)
        if (issued_v[s] > 0) mbar_wait(&sm.v_full[s], (issued_v[s] - 1) & 1, p.wait_ns);
    }
    if (warp == kWarpMma && lane == 0 && mma_issued) {
      umma_commit(&sm.mma_fin);
      mbar_wait(&sm.mma_fin, 0, p.wait_ns);
    }
  }
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
size_t smem_bytes_for() {
  // +1024 for manual alignment; at least 120 KB so that two CTAs never
  // share an SM (each CTA holds all 512 TMEM columns).
  size_t s = sizeof(PrefillSmem<D>) + 1024;
  return s < 120 * 1024 ? 120 * 1024 : s;
}

template <int D>
cudaError_t launch_d(const PrefillArgs& a, const DeviceGuard& g, cudaStream_t stream) {
  KernelParams kp;
  kp.lse = a.lse;
  kp.status = g.status;
  kp.wait_ns = g.wait_ns;
  kp.Hq = a.Hq;
  kp.Hkv = a.Hkv;
  kp.Nq = a.Nq;
  kp.Nk = a.Nk;
  kp.group = a.Hq / a.Hkv;
  kp.n_qtiles = (a.Nq + kBM - 1) / kBM;
  kp.causal = a.causal;
  kp.scale_log2 = a.scale * 1.4426950408889634f;
  const size_t smem = smem_bytes_for<D>();
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(kp.n_qtiles, a.Hq, a.B);
  prefill_kernel<D><<<grid, kThreads, smem, stream>>>(*a.tm_q, *a.tm_k, *a.tm_v, *a.tm_o, kp);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_smem_bytes(int d) { return d == 64 ? smem_bytes_for<64>() : smem_bytes_for<128>(); }

cudaError_t launch_prefill(const PrefillArgs& a, const DeviceGuard& g, cudaStream_t stream) {
  if (a.d == 64) return launch_d<64>(a, g, stream);
  return launch_d<128>(a, g, stream);
}

}  // namespace exattn
