// Attention backward for sm_103a on the tensor cores: dQ, dK, dV from dO and
// the forward's output O and log-sum-exp ("Kernel Fusion, Softmax, and
// Attention" page: training runs a different schedule of the same attention
// equation).  With P_ij = exp(s_ij - lse_i):
//   D_i   = sum_t dO_it O_it                (= sum_j P_ij dP_ij)
//   dP_ij = <dO_i, v_j>,  dS_ij = P_ij (dP_ij - D_i)
//   dV_j  = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,
//   dQ_i  = scale sum_j dS_ij k_j
// P and dS are recomputed tile by tile from Q, K and the saved LSE, never
// stored.  Kernels (no atomics, deterministic), in launch order:
//   * bwd_tc_kernel<D, false> (dQ pass): a CTA holds a 128-row query tile of
//     Q, dO and O and streams 64-key tiles of K and V; its elementwise warps
//     first form D for their rows from dO and O in shared memory and write it
//     for the dK/dV pass; then S = Q K^T, dP = dO V^T, dS = P (dP - D),
//     dQ += dS K;
//   * bwd_tc_kernel<D, true> (dK/dV pass): a CTA holds one 128-key block of
//     K and V in shared memory and streams the 64-row query tiles of one
//     query head that the mask leaves through a 4-stage TMA ring.  Per tile
//     the tensor core forms S^T = K Q^T and dP^T = V dO^T (M128 N64) into a
//     double-buffered pair of TMEM regions; eight elementwise warps (thread =
//     key = TMEM lane, two warps per lane quarter, one per half of the query
//     columns) turn them into P^T and dS^T = P^T (dP^T - D), written back to
//     TMEM as bf16 over their own fp32 columns; then dV += P^T dO and
//     dK += dS^T Q accumulate in TMEM with A read from TMEM and dO, Q
//     MN-major from shared memory.  One query head per KV head writes dK, dV
//     directly; with GQA the G query heads of a KV head run as one cluster
//     of G CTAs (G = 2, 4 or 8): each stages its dK, dV accumulators in its
//     own shared memory and sums 128/G rows of all G over distributed shared
//     memory, in head order; other group sizes write fp32 partials that
//     bwd_reduce_kernel sums in head order.
// Warp roles (320 threads): warps 0-7 elementwise, warp 8 TMA producer,
// warp 9 tcgen05 issuer (warp-uniform loop, one elected lane issues) and
// owner of the TMEM allocation.  Every wait is bounded; a wait that runs
// out sets the device status word, drains what is in flight, frees TMEM and
// returns.
#include <cuda_bf16.h>

#include "launch.h"
#include "ptx.cuh"

namespace exattn {
namespace {

constexpr int kThreads = 320;
constexpr int kWarpLoad = 8;
constexpr int kWarpMma = 9;
constexpr int kStatRows = 128;   // rows of a stationary tile (= TMEM lanes)
constexpr int kStreamRows = 64;  // rows of a streamed tile (= columns of S, dP)
constexpr int kStages = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kBufCol = 256;  // product buffers: 256 + 128 b; the second product at +64
constexpr uint32_t kStatSub = kStatRows * 128;      // one 64-column sub-tile, 128 rows (16 KB)
constexpr uint32_t kStreamSub = kStreamRows * 128;  // one 64-column sub-tile, 64 rows (8 KB)
constexpr float kLog2e = 1.4426950408889634f;

template <int D, bool KV>
struct alignas(1024) BwdSmem {
  uint8_t stat[2][D / 64][kStatSub];              // K, V (dK/dV pass) or Q, dO (dQ pass)
  uint8_t ring[kStages][2][D / 64][kStreamSub];   // Q, dO (dK/dV pass) or K, V (dQ pass)
  uint8_t otile[KV ? 1 : D / 64][KV ? 16 : kStatSub];  // dQ pass: O, for D = rowsum(dO * O)
  uint64_t stat_full, full[kStages], empty[kStages], s_full[2], p_full[2], acc_done, fin;
  uint32_t tmem_base;
  uint32_t abort_flag;
};

struct BwdParams {
  const float* lse;      // [B*Hq, Nq], natural log
  float* dsum;           // [B*Hq, Nq]: D, written by the dQ pass, read by the dK/dV pass
  __nv_bfloat16* out0;   // dK (dK/dV pass, one query head per KV head) or dQ
  __nv_bfloat16* out1;   // dV (dK/dV pass, one query head per KV head)
  float* part;           // dK/dV pass with GQA: partials [G][B*Hkv][Nk][D] of dK, then of dV
  unsigned int* status;
  unsigned long long wait_ns;
  int Hq, Hkv, Nq, Nk, causal, n_bh, n_tiles;
  int cluster;           // dK/dV pass: G when the G query heads of a KV head form a cluster, else 0
  float scale, scale_log2;
};

// Cluster-wide barrier: every thread of every CTA of the cluster arrives;
// release / acquire order the shared-memory writes before it with the
// distributed-shared-memory reads after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __noinline__ bool bwd_wait_slow(uint64_t* bar, uint32_t parity, unsigned long long wait_ns,
                                           unsigned int* status, uint32_t* abort_flag) {
  volatile uint32_t* ab = abort_flag;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*ab) return false;
    if (globaltimer_ns() - t0 > wait_ns) {
      atomicOr(status, 1u);  // EXATTN_DEVICE_TIMEOUT_BIT
      *ab = 1u;
      return false;
    }
  }
}

__device__ __forceinline__ bool bwd_wait(uint64_t* bar, uint32_t parity, const BwdParams& p, uint32_t* ab) {
  if (mbar_try_wait(bar, parity)) return true;
  return bwd_wait_slow(bar, parity, p.wait_ns, p.status, ab);
}

// Which tiles a CTA works on.  KV: a 128-key block of one query head and the
// 64-row query tiles [first, first + count) that see any of its keys.  Q: a
// 128-row query tile and the 64-key tiles [0, count) that it sees.
struct Work {
  int bh, tile;      // (b * Hq + hq), stationary tile index
  int splane, srow;  // stationary tensor plane and first row
  int rplane, first, count;
};

template <bool KV>
__device__ __forceinline__ Work work_of(int cta, const BwdParams& p) {
  Work w;
  w.bh = cta % p.n_bh;
  const int hq = w.bh % p.Hq, b = w.bh / p.Hq;
  const int kv_plane = b * p.Hkv + hq / (p.Hq / p.Hkv);
  const long long shift = static_cast<long long>(p.Nk) - p.Nq;
  if (KV) {
    w.tile = cta / p.n_bh;  // key block; under the mask the first ones see the most queries
    w.splane = kv_plane;
    w.srow = w.tile * kStatRows;
    w.rplane = w.bh;
    const int n_q = (p.Nq + kStreamRows - 1) / kStreamRows;
    int first = 0;
    if (p.causal) {  // query rows i see key j iff j <= i + shift
      const long long row = static_cast<long long>(w.srow) - shift;
      first = row <= 0 ? 0 : static_cast<int>(min(row / kStreamRows, static_cast<long long>(n_q)));
    }
    w.first = first;
    w.count = n_q - first;
  } else {
    w.tile = p.n_tiles - 1 - cta / p.n_bh;  // query tile; the last ones see the most keys
    w.splane = w.bh;
    w.srow = w.tile * kStatRows;
    w.rplane = kv_plane;
    w.first = 0;
    int n_k = (p.Nk + kStreamRows - 1) / kStreamRows;
    if (p.causal) {
      const long long last = static_cast<long long>(w.srow) + kStatRows - 1 + shift;  // last key seen
      n_k = last < 0 ? 0 : static_cast<int>(min(last / kStreamRows + 1, static_cast<long long>(n_k)));
    }
    w.count = n_k;
  }
  return w;
}

template <int D, bool KV>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_s0, const __grid_constant__ CUtensorMap tm_s1,
                  const __grid_constant__ CUtensorMap tm_r0, const __grid_constant__ CUtensorMap tm_r1,
                  const __grid_constant__ CUtensorMap tm_o, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  BwdSmem<D, KV>& sm = *reinterpret_cast<BwdSmem<D, KV>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Work w = work_of<KV>(blockIdx.x, p);

  if (warp == kWarpLoad && lane == 0) {
    tma_prefetch_desc(&tm_s0);
    tma_prefetch_desc(&tm_s1);
    tma_prefetch_desc(&tm_r0);
    tma_prefetch_desc(&tm_r1);
    if (!KV) tma_prefetch_desc(&tm_o);
    mbar_init(&sm.stat_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.p_full[b], 8);
    }
    mbar_init(&sm.acc_done, 1);
    mbar_init(&sm.fin, 1);
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
  const int n = w.count;

  int loads_issued = 0;   // producer: streamed tiles issued
  bool stat_issued = false;
  bool mma_issued = false;

  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ producer
    // the dQ pass needs its tiles for D even when no key tile is left
    if (lane == 0 && (n > 0 || !KV)) {
      const uint64_t keep = l2_policy_evict_last();  // streamed tiles are re-read by other CTAs
      mbar_arrive_expect_tx(&sm.stat_full, (KV ? 2 : 3) * D * kStatRows * 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(sm.stat[0][c], &tm_s0, &sm.stat_full, c * 64, w.srow, w.splane);
        tma_load_3d(sm.stat[1][c], &tm_s1, &sm.stat_full, c * 64, w.srow, w.splane);
        if (!KV) tma_load_3d(sm.otile[c], &tm_o, &sm.stat_full, c * 64, w.srow, w.splane);
      }
      stat_issued = true;
      for (int i = 0; i < n; ++i) {
        const int s = i % kStages;
        if (i >= kStages && !bwd_wait(&sm.empty[s], ((i / kStages) - 1) & 1, p, &sm.abort_flag)) break;
        const int row = (w.first + i) * kStreamRows;
        mbar_arrive_expect_tx(&sm.full[s], 2 * D * kStreamRows * 2);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d_hint(sm.ring[s][0][c], &tm_r0, &sm.full[s], c * 64, row, w.rplane, keep);
          tma_load_3d_hint(sm.ring[s][1][c], &tm_r1, &sm.full[s], c * 64, row, w.rplane, keep);
        }
        loads_issued = i + 1;
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (n > 0) {
      constexpr uint32_t id_prod = idesc_bf16_f32(128, kStreamRows, false, false);
      constexpr uint32_t id_acc = idesc_bf16_f32(128, D, false, true);
      const uint64_t d_s0 = smem_desc(smem_u32(&sm.stat[0][0][0]), 16, 1024, kSwizzle128B);
      const uint64_t d_s1 = smem_desc(smem_u32(&sm.stat[1][0][0]), 16, 1024, kSwizzle128B);
      constexpr uint32_t kStageUnits = 2 * (D / 64) * kStreamSub / 16;
      constexpr uint32_t kSlotUnits = (D / 64) * kStreamSub / 16;
      const uint64_t d_r_k = smem_desc(smem_u32(&sm.ring[0][0][0][0]), 16, 1024, kSwizzle128B);
      const uint64_t d_r_mn = smem_desc(smem_u32(&sm.ring[0][0][0][0]), kStreamSub, 1024, kSwizzle128B);
      auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, bwd_wait(bar, parity, p, &sm.abort_flag));
      };
      // products of tile i (ring stage s) into buffer b
      auto products = [&](int s, int b) {
        const uint32_t col = kBufCol + 128u * b;
        const uint64_t r0 = d_r_k + static_cast<uint64_t>(s * kStageUnits);
        const uint64_t r1 = r0 + kSlotUnits;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t oa = (kk / 4) * (kStatSub / 16) + (kk % 4) * 2;
          const uint32_t ob = (kk / 4) * (kStreamSub / 16) + (kk % 4) * 2;
          umma_bf16_ss_warp(tmem + col, d_s0 + oa, r0 + ob, id_prod, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t oa = (kk / 4) * (kStatSub / 16) + (kk % 4) * 2;
          const uint32_t ob = (kk / 4) * (kStreamSub / 16) + (kk % 4) * 2;
          umma_bf16_ss_warp(tmem + col + 64, d_s1 + oa, r1 + ob, id_prod, kk > 0 ? 1u : 0u);
        }
        umma_commit_warp(&sm.s_full[b]);
      };
      // accumulations of tile i (stage s, buffer b); first = the CTA's first tile
      auto accumulate = [&](int s, int b, bool first) {
        const uint32_t col = kBufCol + 128u * b;
        const uint64_t r0 = d_r_mn + static_cast<uint64_t>(s * kStageUnits);
        const uint64_t r1 = r0 + kSlotUnits;
#pragma unroll
        for (int kk = 0; kk < kStreamRows / 16; ++kk) {
          const uint32_t a_off = (kk / 2) * 32 + (kk % 2) * 8;  // packed columns of rows 16kk..
          const uint32_t acc = (first && kk == 0) ? 0u : 1u;
          if (KV) {
            // dV += P^T dO, dK += dS^T Q
            umma_bf16_ts_warp(tmem + 0, tmem + col + a_off, r1 + kk * 128, id_acc, acc);
            umma_bf16_ts_warp(tmem + D, tmem + col + 64 + a_off, r0 + kk * 128, id_acc, acc);
          } else {
            // dQ += dS K
            umma_bf16_ts_warp(tmem + 0, tmem + col + a_off, r0 + kk * 128, id_acc, acc);
          }
        }
        umma_commit_warp(&sm.empty[s]);
      };
      bool ok = wait_all(&sm.stat_full, 0);
      for (int i = 0; ok && i < n; ++i) {
        const int s = i % kStages, b = i & 1;
        if (!(ok = wait_all(&sm.full[s], (i / kStages) & 1))) break;
        tc_fence_after_sync();
        mma_issued = true;
        products(s, b);
        if (i >= 1) {
          const int j = i - 1;
          if (!(ok = wait_all(&sm.p_full[j & 1], (j >> 1) & 1))) break;
          tc_fence_after_sync();
          accumulate(j % kStages, j & 1, j == 0);
        }
      }
      if (ok) {
        const int j = n - 1;
        if ((ok = wait_all(&sm.p_full[j & 1], (j >> 1) & 1))) {
          tc_fence_after_sync();
          accumulate(j % kStages, j & 1, j == 0);
          umma_commit_warp(&sm.acc_done);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ elementwise warps
    const int quarter = warp & 3;  // TMEM lanes 32 quarter ..
    const int half = warp >> 2;    // columns 32 half .. of the 64 streamed rows
    const int r = quarter * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const long long shift = static_cast<long long>(p.Nk) - p.Nq;
    const int row = w.srow + r;  // key (dK/dV pass) or query row (dQ pass) of this thread
    const size_t lrow0 = static_cast<size_t>(w.bh) * p.Nq;
    float row_lse2 = 0.f, row_d = 0.f;
    bool ok = true;
    if constexpr (!KV) {
      // D of this thread's query row from the dO and O tiles (rows past Nq
      // read as zero); written once, by the first half, for the dK/dV pass
      if (row < p.Nq) row_lse2 = p.lse[lrow0 + row] * kLog2e;
      ok = __all_sync(0xffffffffu, bwd_wait(&sm.stat_full, 0, p, &sm.abort_flag));
      if (ok) {
        const uint8_t* dob = &sm.stat[1][0][0];
        const uint8_t* ob = &sm.otile[0][0];
        float acc = 0.f;
#pragma unroll
        for (int sub = 0; sub < D / 64; ++sub)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t off = sub * kStatSub + (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4);
            float fo[8], fd[8];
            unpack_bf16x8(*reinterpret_cast<const uint4*>(ob + off), fo);
            unpack_bf16x8(*reinterpret_cast<const uint4*>(dob + off), fd);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc = fmaf(fd[e], fo[e], acc);
          }
        row_d = acc;
        if (half == 0 && row < p.Nq) p.dsum[lrow0 + row] = acc;
      }
    }
    for (int i = 0; i < n; ++i) {
      const int b = i & 1;
      const int c0 = (w.first + i) * kStreamRows + half * 32;  // first streamed row of this half
      float col_lse2 = 0.f, col_d = 0.f;  // dK/dV pass: query c0 + lane
      if (KV && c0 + lane < p.Nq) {
        col_lse2 = p.lse[lrow0 + c0 + lane] * kLog2e;
        col_d = p.dsum[lrow0 + c0 + lane];
      }
      if (!__all_sync(0xffffffffu, bwd_wait(&sm.s_full[b], (i >> 1) & 1, p, &sm.abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t col = kBufCol + 128u * b + half * 32;
      uint32_t sv[32], dpv[32];
      tmem_ld_32x32b_x32(t_lane + col, sv);
      tmem_ld_32x32b_x32(t_lane + col + 64, dpv);
      tmem_ld_wait();
      uint32_t pk[16], dsk[16];
      // Is every element of this warp's 32 x 32 block visible and in range?
      // Then no element needs a mask test.
      const long long r_lo = w.srow + quarter * 32, r_hi = r_lo + 31;  // this warp's rows
      const long long c_lo = c0, c_hi = c0 + 31;                       // this warp's columns
      const bool interior = KV ? (r_hi < p.Nk && c_hi < p.Nq && (!p.causal || r_hi <= c_lo + shift))
                               : (r_hi < p.Nq && c_hi < p.Nk && (!p.causal || c_hi <= r_lo + shift));
      if (interior) {
        const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float l2a = KV ? __shfl_sync(0xffffffffu, col_lse2, c) : row_lse2;
          const float l2b = KV ? __shfl_sync(0xffffffffu, col_lse2, c + 1) : row_lse2;
          const float da = KV ? __shfl_sync(0xffffffffu, col_d, c) : row_d;
          const float db = KV ? __shfl_sync(0xffffffffu, col_d, c + 1) : row_d;
          const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sc2, f2_pack(-l2a, -l2b));
          float x0, x1;
          f2_unpack(x2, x0, x1);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          const uint64_t t2 = f2_add(f2_pack(__uint_as_float(dpv[c]), __uint_as_float(dpv[c + 1])), f2_pack(-da, -db));
          float d0, d1;
          f2_unpack(f2_mul(f2_pack(p0, p1), t2), d0, d1);
          pk[c / 2] = pack_bf16x2(p0, p1);
          dsk[c / 2] = pack_bf16x2(d0, d1);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float pr[2], ds[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int cc = c + e;
            // (key, query) of this element
            const long long key = KV ? row : c0 + cc;
            const long long qry = KV ? c0 + cc : row;
            const float l2 = KV ? __shfl_sync(0xffffffffu, col_lse2, cc) : row_lse2;
            const float dd = KV ? __shfl_sync(0xffffffffu, col_d, cc) : row_d;
            const bool vis = key < p.Nk && qry < p.Nq && (!p.causal || key <= qry + shift);
            const float pe = vis ? ex2_approx(__uint_as_float(sv[cc]) * p.scale_log2 - l2) : 0.f;
            pr[e] = pe;
            ds[e] = vis ? pe * (__uint_as_float(dpv[cc]) - dd) : 0.f;
          }
          pk[c / 2] = pack_bf16x2(pr[0], pr[1]);
          dsk[c / 2] = pack_bf16x2(ds[0], ds[1]);
        }
      }
      // bf16 P^T (dK/dV pass) over this half's own first 16 S columns, bf16
      // dS over its own first 16 dP columns (dK/dV pass) or S columns (dQ pass)
      if (KV) {
        tmem_st_32x32b_x16(t_lane + col, pk);
        tmem_st_32x32b_x16(t_lane + col + 64, dsk);
      } else {
        tmem_st_32x32b_x16(t_lane + col, dsk);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full[b]);
    }
    // ---------------------------------------------------------- epilogue
    if (ok) {
      if (n > 0) {
        if (!__all_sync(0xffffffffu, bwd_wait(&sm.acc_done, 0, p, &sm.abort_flag))) ok = false;
        tc_fence_after_sync();
      }
    }
    if (ok) {
      constexpr int kHalf = D / 2;  // accumulator columns of this thread
      const int col0 = half * kHalf;
      const int n_acc = KV ? 2 : 1;
#pragma unroll 1
      for (int a = 0; a < n_acc; ++a) {
        uint32_t v[kHalf];
        if (n > 0) {
#pragma unroll
          for (int c = 0; c < kHalf / 32; ++c)
            tmem_ld_32x32b_x32(t_lane + a * D + col0 + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * c]));
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < kHalf; ++e) v[e] = 0u;
        }
        // dK/dV pass: a = 0 is dV, a = 1 is dK (times scale); dQ pass: dQ (times scale)
        const float mul = (KV && a == 0) ? 1.f : p.scale;
        const int lim = KV ? p.Nk : p.Nq;
        if (KV && p.cluster > 0) {
          // staged for the cluster's sum in the teardown (row stride D + 4 floats)
          float* st = reinterpret_cast<float*>(&sm.stat[0][0][0]) + (a * kStatRows + r) * (D + 4) + col0;
#pragma unroll
          for (int c = 0; c < kHalf / 4; ++c)
            *reinterpret_cast<float4*>(st + 4 * c) = make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                                                                 __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3]));
        } else if (row < lim) {
          if (!KV || p.part == nullptr) {
            const size_t plane = KV ? static_cast<size_t>(w.splane) : static_cast<size_t>(w.bh);
            __nv_bfloat16* dst = (KV && a == 0) ? p.out1 : p.out0;
            uint4* o = reinterpret_cast<uint4*>(dst + (plane * lim + row) * D + col0);
#pragma unroll
            for (int c = 0; c < kHalf / 8; ++c)
              o[c] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * c]) * mul, __uint_as_float(v[8 * c + 1]) * mul),
                                pack_bf16x2(__uint_as_float(v[8 * c + 2]) * mul, __uint_as_float(v[8 * c + 3]) * mul),
                                pack_bf16x2(__uint_as_float(v[8 * c + 4]) * mul, __uint_as_float(v[8 * c + 5]) * mul),
                                pack_bf16x2(__uint_as_float(v[8 * c + 6]) * mul, __uint_as_float(v[8 * c + 7]) * mul));
          } else {
            // fp32 partials of query head hq % G: [g][B*Hkv][Nk][D] for dK, then [G + g] for dV
            const int G = p.Hq / p.Hkv;
            const size_t plane_elems = static_cast<size_t>(p.n_bh / G) * p.Nk * D;
            const int g = (w.bh % p.Hq) % G;
            float* dst = p.part + static_cast<size_t>(a == 0 ? G + g : g) * plane_elems +
                         (static_cast<size_t>(w.splane) * p.Nk + row) * D + col0;
            float4* o = reinterpret_cast<float4*>(dst);
#pragma unroll
            for (int c = 0; c < kHalf / 4; ++c)
              o[c] = make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                                 __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3]));
          }
        }
      }
    }
    tc_fence_before_sync();
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  const bool aborted = *reinterpret_cast<volatile uint32_t*>(&sm.abort_flag) != 0u;
  if (aborted) {
    // Drain what is still in flight before the CTA's memory goes away.
    if (warp == kWarpLoad && lane == 0) {
      if (stat_issued) mbar_wait(&sm.stat_full, 0, p.wait_ns);
      for (int i = loads_issued - kStages; i < loads_issued; ++i)
        if (i >= 0) mbar_wait(&sm.full[i % kStages], (i / kStages) & 1, p.wait_ns);
    }
    if (warp == kWarpMma && lane == 0 && mma_issued) {
      umma_commit(&sm.fin);
      mbar_wait(&sm.fin, 0, p.wait_ns);
    }
  }
  __syncthreads();
  if (KV && p.cluster > 0) {
    // dK, dV of this key block: the sum over the cluster's G query heads,
    // in head (cluster rank) order.  Rank k sums rows [128/G k, 128/G (k+1)).
    cluster_sync_all();
    uint32_t rank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const int G = p.cluster;
    const int R = kStatRows / G;
    const uint32_t base = smem_u32(&sm.stat[0][0][0]);
    const int items = 2 * R * (D / 4);  // (accumulator, row, 4 columns)
    for (int it = threadIdx.x; it < items; it += kThreads) {
      const int c4 = it % (D / 4);
      const int rl = (it / (D / 4)) % R;
      const int a = it / (R * (D / 4));  // 0: dV, 1: dK
      const int rr = static_cast<int>(rank) * R + rl;
      const int key = w.srow + rr;
      const uint32_t off = base + static_cast<uint32_t>(((a * kStatRows + rr) * (D + 4) + 4 * c4) * 4);
      float x = 0.f, y = 0.f, z = 0.f, u = 0.f;
      for (int k = 0; k < G; ++k) {
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(off), "r"(k));
        float4 f;
        asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w) : "r"(remote) : "memory");
        x += f.x; y += f.y; z += f.z; u += f.w;
      }
      if (key < p.Nk) {
        const float mul = a == 0 ? 1.f : p.scale;
        __nv_bfloat16* dst = a == 0 ? p.out1 : p.out0;
        *reinterpret_cast<uint2*>(dst + (static_cast<size_t>(w.splane) * p.Nk + key) * D + 4 * c4) =
            make_uint2(pack_bf16x2(x * mul, y * mul), pack_bf16x2(z * mul, u * mul));
      }
    }
    cluster_sync_all();  // no CTA leaves while a peer may still read its shared memory
  }
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// dK = scale * sum_g partial_g, dV = sum_g partial_g, in head order.
template <int D>
__global__ void __launch_bounds__(256) bwd_reduce_kernel(const float* part, __nv_bfloat16* dk,
                                                         __nv_bfloat16* dv, long long n_elems, int G,
                                                         float scale) {
  const long long i = (static_cast<long long>(blockIdx.x) * 256 + threadIdx.x) * 4;
  if (i >= n_elems) return;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f), c = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int gi = 0; gi < G; ++gi) {
    const float4 x = *reinterpret_cast<const float4*>(part + gi * n_elems + i);
    const float4 y = *reinterpret_cast<const float4*>(part + (G + gi) * n_elems + i);
    a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
    c.x += y.x; c.y += y.y; c.z += y.z; c.w += y.w;
  }
  *reinterpret_cast<uint2*>(dk + i) = make_uint2(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale));
  *reinterpret_cast<uint2*>(dv + i) = make_uint2(pack_bf16x2(c.x, c.y), pack_bf16x2(c.z, c.w));
}

// +1024 for manual alignment; at least 120 KB so that two CTAs never share
// an SM (each holds all 512 TMEM columns).
template <int D, bool KV>
constexpr size_t bwd_smem_bytes() {
  return sizeof(BwdSmem<D, KV>) + 1024 < 120 * 1024 ? 120 * 1024 : sizeof(BwdSmem<D, KV>) + 1024;
}

template <int D>
cudaError_t launch_bwd_d(const BwdArgs& a, const DeviceGuard& g, cudaStream_t stream) {
  BwdParams p;
  p.lse = a.lse;
  p.dsum = a.dsum;
  p.status = g.status;
  p.wait_ns = g.wait_ns;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.causal = a.causal;
  p.n_bh = a.B * a.Hq;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.cluster = 0;
  constexpr int smem_kv = static_cast<int>(bwd_smem_bytes<D, true>());
  constexpr int smem_q = static_cast<int>(bwd_smem_bytes<D, false>());
  static std::atomic<int> set_kv[64] = {}, set_q[64] = {};
  cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(bwd_tc_kernel<D, true>), smem_kv, set_kv);
  if (e != cudaSuccess) return e;
  e = smem_limit_once(reinterpret_cast<const void*>(bwd_tc_kernel<D, false>), smem_q, set_q);
  if (e != cudaSuccess) return e;
  // dQ pass first: it writes D, which the dK/dV pass reads
  if (a.Nq > 0) {
    BwdParams pq = p;
    pq.out0 = static_cast<__nv_bfloat16*>(a.dq);
    pq.out1 = nullptr;
    pq.part = nullptr;
    pq.n_tiles = (a.Nq + kStatRows - 1) / kStatRows;
    const long long grid = static_cast<long long>(pq.n_tiles) * pq.n_bh;
    bwd_tc_kernel<D, false><<<static_cast<unsigned>(grid), kThreads, smem_q, stream>>>(
        *a.tm_q128, *a.tm_do128, *a.tm_k64, *a.tm_v64, *a.tm_o128, pq);
  }
  const int G = a.Hq / a.Hkv;
  if (a.Nk > 0) {
    BwdParams pk = p;
    pk.out0 = static_cast<__nv_bfloat16*>(a.dk);
    pk.out1 = static_cast<__nv_bfloat16*>(a.dv);
    bool clustered = G == 2 || G == 4 || G == 8;
    if (clustered) {
      // the cluster shape must fit the device at least once (G SMs of one
      // GPC with this much shared memory each); else the partial-sum path
      static std::atomic<int> fits[64][4] = {};  // per device and G = 2, 4, 8: 0 unknown, 1 yes, 2 no
      int dev = 0;
      if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
      const int gi = G == 2 ? 0 : (G == 4 ? 1 : 2);
      int f = fits[dev][gi].load(std::memory_order_acquire);
      if (f == 0) {
        cudaLaunchConfig_t probe = {};
        probe.gridDim = dim3(static_cast<unsigned>(G));
        probe.blockDim = dim3(kThreads);
        probe.dynamicSmemBytes = smem_kv;
        cudaLaunchAttribute pa[1];
        pa[0].id = cudaLaunchAttributeClusterDimension;
        pa[0].val.clusterDim.x = G;
        pa[0].val.clusterDim.y = 1;
        pa[0].val.clusterDim.z = 1;
        probe.attrs = pa;
        probe.numAttrs = 1;
        int n_clusters = 0;
        const cudaError_t qe =
            cudaOccupancyMaxActiveClusters(&n_clusters, bwd_tc_kernel<D, true>, &probe);
        f = (qe == cudaSuccess && n_clusters > 0) ? 1 : 2;
        if (qe != cudaSuccess) (void)cudaGetLastError();  // a refused query leaves no sticky error
        fits[dev][gi].store(f, std::memory_order_release);
      }
      clustered = f == 1;
    }
    pk.part = (G > 1 && !clustered) ? a.part : nullptr;
    pk.cluster = clustered ? G : 0;
    pk.n_tiles = (a.Nk + kStatRows - 1) / kStatRows;
    const long long grid = static_cast<long long>(pk.n_tiles) * pk.n_bh;
    if (clustered) {
      // the G CTAs of a (key block, KV head) are consecutive: b * Hq + hkv * G + g
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(grid));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = smem_kv;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = G;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&cfg, bwd_tc_kernel<D, true>, *a.tm_k128, *a.tm_v128, *a.tm_q64, *a.tm_do64,
                             *a.tm_k128, pk);
      if (e != cudaSuccess) return e;
    } else {
      bwd_tc_kernel<D, true><<<static_cast<unsigned>(grid), kThreads, smem_kv, stream>>>(
          *a.tm_k128, *a.tm_v128, *a.tm_q64, *a.tm_do64, *a.tm_k128, pk);
    }
    if (G > 1 && !clustered) {
      const long long n = static_cast<long long>(a.B) * a.Hkv * a.Nk * D;
      bwd_reduce_kernel<D><<<static_cast<unsigned>((n / 4 + 255) / 256), 256, 0, stream>>>(
          a.part, static_cast<__nv_bfloat16*>(a.dk), static_cast<__nv_bfloat16*>(a.dv), n, G, a.scale);
    }
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, const DeviceGuard& g, cudaStream_t stream) {
  return a.d == 64 ? launch_bwd_d<64>(a, g, stream) : launch_bwd_d<128>(a, g, stream);
}

}  // namespace exattn
