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
//   * bwd_tc_kernel<D, false> (dQ pass): a unit is a 128-row query tile of
//     one head.  Its Q, dO and O tiles come into shared memory; the MMA warp
//     copies Q and dO into TMEM (tcgen05.cp), where they are the A operands
//     of S = Q K^T and dP = dO V^T (M128 N64, B = the streamed 64-key K and
//     V tiles of a 4-stage TMA ring), so the tensor core reads only the
//     streamed tiles from shared memory.  The elementwise warps form D for
//     their rows from dO and O (each half of the warps over its half of the
//     columns) and write (lse * log2 e, D) for the dK/dV pass.  dS =
//     P (dP - D) goes back to TMEM as bf16 and dQ += dS K accumulates in
//     TMEM.  dQ leaves through the O tile's slot: staged there in bf16 and
//     written by a TMA store;
//   * bwd_tc_kernel<D, true> (dK/dV pass): a unit is a 128-key block of one
//     query head.  K and V stay in shared memory; the 64-row query tiles of
//     that head that the mask leaves stream through the ring, each with its
//     queries' (lse * log2 e, D) pairs.  Per tile the tensor core forms
//     S^T = K Q^T and dP^T = V dO^T (M128 N64) into a double-buffered pair
//     of TMEM regions; eight elementwise warps (thread = key = TMEM lane, two
//     warps per lane quarter, one per half of the query columns, the pairs
//     read as shared-memory broadcasts) turn them into P^T and
//     dS^T = P^T (dP^T - D), written back to TMEM as bf16 over their own
//     fp32 columns; then dV += P^T dO and dK += dS^T Q accumulate in TMEM
//     with A read from TMEM and dO, Q MN-major from shared memory.  With one
//     query head per KV head it writes dK, dV directly; with GQA each query
//     head writes fp32 partials (32-byte stores) that bwd_reduce_kernel sums
//     in head order.
// The dK/dV pass and the GQA sum are programmatic dependent launches: each
// grid may start on SMs that the previous one has left while that one's
// last CTAs finish, and waits for its results where it reads them.
// Both passes are persistent (one CTA per SM, grid = min(units, SMs)); CTA
// c takes unit r*G + c in even rounds r and r*G + G-1-c in odd ones, units
// numbered heaviest first under the causal mask.  A CTA's TMA ring, product
// buffers and accumulators run on across its units: the next unit's
// stationary tiles load while the current one drains, and its first
// products are queued before the previous unit's epilogue is done.
// Warp roles (352 threads): warps 0-7 elementwise, warp 8 TMA producer,
// warp 9 tcgen05 issuer (warp-uniform loop, one elected lane issues) and
// owner of the TMEM allocation, warp 10 the dQ pass's TMA stores.  Every
// wait is bounded; a wait that runs out sets the device status word, drains
// what is in flight, frees TMEM and returns.
#include <cuda_bf16.h>

#include "launch.h"
#include "ptx.cuh"

namespace exattn {
namespace {

constexpr int kThreads = 352;
constexpr int kWarpLoad = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpStore = 10;  // dQ pass: TMA stores of dQ
constexpr int kStatRows = 128;   // rows of a stationary tile (= TMEM lanes)
constexpr int kStreamRows = 64;  // rows of a streamed tile (= columns of S, dP)
constexpr int kStages = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kBufCol = 256;  // product buffers: 256 + 128 b; the second product at +64
// dQ pass: Q and dO of the query tile as TMEM A operands (two bf16 a column)
// at columns 128 and 128 + d/2, between the dQ accumulator and the buffers
constexpr uint32_t kQCol = 128;
constexpr uint32_t kStatSub = kStatRows * 128;      // one 64-column sub-tile, 128 rows (16 KB)
constexpr uint32_t kStreamSub = kStreamRows * 128;  // one 64-column sub-tile, 64 rows (8 KB)
constexpr float kLog2e = 1.4426950408889634f;

template <int D, bool KV>
struct alignas(1024) BwdSmem {
  uint8_t stat[2][D / 64][kStatSub];              // K, V (dK/dV pass) or Q, dO (dQ pass)
  uint8_t ring[kStages][2][D / 64][kStreamSub];   // Q, dO (dK/dV pass) or K, V (dQ pass)
  uint8_t otile[KV ? 1 : D / 64][KV ? 16 : kStatSub];  // dQ pass: O, for D = rowsum(dO * O)
  float dpart[KV ? 1 : 2][KV ? 1 : kStatRows];          // dQ pass: D of each half of the columns
  alignas(128) float ldp[KV ? kStages : 1][KV ? 2 * kStreamRows : 4];  // dK/dV pass: (lse * log2 e, D) of the streamed queries
  uint64_t stat_full, stat_free, full[kStages], empty[kStages], s_full[2], p_full[2], acc_done, acc_free, fin;
  uint64_t a_free;          // dQ pass: the unit's last products have read the TMEM copies of Q and dO
  uint64_t dpart_full;      // dQ pass: both halves' shares of D written
  uint64_t dq_staged;       // dQ pass: the tiles read (first phase), then each unit's dQ staged
  uint32_t tmem_base;
  uint32_t abort_flag;
};

struct BwdParams {
  const float* lse;      // [B*Hq, Nq], natural log
  float* ldp;            // [B*Hq][nq_pad][2]: (lse * log2 e, D), written by the dQ pass, loaded by the dK/dV pass
  __nv_bfloat16* out0;   // dK (dK/dV pass, one query head per KV head) or dQ
  __nv_bfloat16* out1;   // dV (dK/dV pass, one query head per KV head)
  float* part;           // dK/dV pass with GQA: partials [G][B*Hkv][Nk][D] of dK, then of dV
  unsigned int* status;
  unsigned long long wait_ns;
  int Hq, Hkv, Nq, Nk, causal, n_bh, n_tiles, nq_pad;
  float scale, scale_log2;
};

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

// The tiles of work unit u.  KV: a 128-key block of one query head and the
// 64-row query tiles [first, first + count) that see any of its keys.  Q: a
// 128-row query tile and the 64-key tiles [0, count) that it sees.  Units
// are numbered heaviest first under the causal mask.
struct Work {
  int bh, tile;      // (b * Hq + hq), stationary tile index
  int splane, srow;  // stationary tensor plane and first row
  int rplane, first, count;
};

// a = b = +0 unless lo <= c < hi (one predicate, two selects)
__device__ __forceinline__ void keep_in_range(int c, int lo, int hi, uint32_t& a, uint32_t& b) {
  asm("{\n\t.reg .pred q;\n\t"
      "setp.ge.s32 q, %2, %3;\n\t"
      "setp.lt.and.s32 q, %2, %4, q;\n\t"
      "selp.b32 %0, %0, 0, q;\n\t"
      "selp.b32 %1, %1, 0, q;\n\t}"
      : "+r"(a), "+r"(b) : "r"(c), "r"(lo), "r"(hi));
}

// P and dS of one thread's 32 elements (one row of a warp's 32 x 32
// block): p = 2^(s * scale * log2e - lse * log2e), ds = p (dp - D).  The
// row's lse and D are per thread in the dQ pass (row = query) and per column
// in the dK/dV pass (row = key): there the (lse * log2e, D) pairs of the 32
// columns, in shared memory, read as broadcasts.  kMasked: the elements
// outside [lo, hi) become +0.
template <bool KV, bool kMasked>
__device__ __forceinline__ void bwd_block(const uint32_t (&sv)[32], const uint32_t (&dpv)[32], float scale_log2,
                                          float row_lse2, float row_d, const float* cols, int lo, int hi,
                                          uint32_t (&pk)[16], uint32_t (&dsk)[16]) {
  const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    float l2a = row_lse2, l2b = row_lse2, da = row_d, db = row_d;
    if constexpr (KV) {
      const float4 q = *reinterpret_cast<const float4*>(cols + 2 * c);
      l2a = q.x;
      da = q.y;
      l2b = q.z;
      db = q.w;
    }
    const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sc2, f2_pack(-l2a, -l2b));
    float x0, x1;
    f2_unpack(x2, x0, x1);
    uint32_t p0 = __float_as_uint(ex2_approx(x0)), p1 = __float_as_uint(ex2_approx(x1));
    const uint64_t t2 = f2_add(f2_pack(__uint_as_float(dpv[c]), __uint_as_float(dpv[c + 1])), f2_pack(-da, -db));
    float d0f, d1f;
    f2_unpack(f2_mul(f2_pack(__uint_as_float(p0), __uint_as_float(p1)), t2), d0f, d1f);
    uint32_t d0 = __float_as_uint(d0f), d1 = __float_as_uint(d1f);
    if constexpr (kMasked) {
      keep_in_range(c, lo, hi, p0, d0);
      keep_in_range(c + 1, lo, hi, p1, d1);
    }
    pk[c / 2] = pack_bf16x2(__uint_as_float(p0), __uint_as_float(p1));
    dsk[c / 2] = pack_bf16x2(__uint_as_float(d0), __uint_as_float(d1));
  }
}

template <bool KV>
__device__ __forceinline__ Work work_of(int u, const BwdParams& p) {
  Work w;
  w.bh = u % p.n_bh;
  const int hq = w.bh % p.Hq, b = w.bh / p.Hq;
  const int kv_plane = b * p.Hkv + hq / (p.Hq / p.Hkv);
  const long long shift = static_cast<long long>(p.Nk) - p.Nq;
  if (KV) {
    w.tile = u / p.n_bh;  // key block; under the mask the first ones see the most queries
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
    w.tile = p.n_tiles - 1 - u / p.n_bh;  // query tile; the last ones see the most keys
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
                  const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_dq,
                  const __grid_constant__ CUtensorMap tm_ldp, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  BwdSmem<D, KV>& sm = *reinterpret_cast<BwdSmem<D, KV>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // The next launch of the backward (the dK/dV pass after the dQ pass, the
  // GQA sum after the dK/dV pass) may be scheduled as soon as every CTA of
  // this grid has started; it takes SMs as this grid's CTAs finish.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_units = p.n_tiles * p.n_bh;
  // Persistent: CTA c takes unit r*G + c (r even) or r*G + G-1-c (r odd) in
  // round r, G = gridDim.x; units are numbered heaviest first.
  auto unit_of = [&](int round) -> int {
    const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    return round * G + ((round & 1) ? (G - 1 - c) : c);
  };

  if (warp == kWarpLoad && lane == 0) {
    tma_prefetch_desc(&tm_s0);
    tma_prefetch_desc(&tm_s1);
    tma_prefetch_desc(&tm_r0);
    tma_prefetch_desc(&tm_r1);
    if (!KV) {
      tma_prefetch_desc(&tm_o);
      tma_prefetch_desc(&tm_dq);
    } else {
      tma_prefetch_desc(&tm_ldp);
    }
    mbar_init(&sm.stat_full, 1);
    // The stationary tiles are released by the MMA warp's commit after a
    // unit's last products (dK/dV pass), or (dQ pass) by two arrivals: the
    // MMA warp's commit after its copies of Q and dO into TMEM, and the
    // store warp's: the O tile's slot stages the previous unit's dQ, written
    // by each elementwise warp over the bytes of O that it has read, and is
    // free once the TMA store has read it.
    mbar_init(&sm.stat_free, KV ? 1 : 2);
    mbar_init(&sm.a_free, 1);
    mbar_init(&sm.dpart_full, 8);
    mbar_init(&sm.dq_staged, 8);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.s_full[b], 1);
      mbar_init(&sm.p_full[b], 8);
    }
    mbar_init(&sm.acc_done, 1);
    mbar_init(&sm.acc_free, 8);
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

  int stat_loads = 0;     // producer: stationary loads issued
  int loads_issued = 0;   // producer: streamed tiles issued (running over units)
  bool mma_issued = false;

  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last();  // streamed tiles are re-read by other CTAs
      bool ok = true;
      bool dq_done = false;  // dK/dV pass: the dQ pass (which writes lse and D pairs) has completed
      for (int round = 0; ok; ++round) {
        const int u = unit_of(round);
        if (u >= n_units) break;
        const Work w = work_of<KV>(u, p);
        // the previous unit's stationary tiles must be released first
        if (stat_loads > 0 && !(ok = bwd_wait(&sm.stat_free, (stat_loads - 1) & 1, p, &sm.abort_flag))) break;
        mbar_arrive_expect_tx(&sm.stat_full, (KV ? 2 : 3) * D * kStatRows * 2);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(sm.stat[0][c], &tm_s0, &sm.stat_full, c * 64, w.srow, w.splane);
          tma_load_3d(sm.stat[1][c], &tm_s1, &sm.stat_full, c * 64, w.srow, w.splane);
          if (!KV) tma_load_3d(sm.otile[c], &tm_o, &sm.stat_full, c * 64, w.srow, w.splane);
        }
        ++stat_loads;
        for (int i = 0; i < w.count; ++i) {
          const int t = loads_issued;
          const int s = t % kStages;
          if (t >= kStages && !(ok = bwd_wait(&sm.empty[s], ((t / kStages) - 1) & 1, p, &sm.abort_flag))) break;
          const int row = (w.first + i) * kStreamRows;
          mbar_arrive_expect_tx(&sm.full[s], 2 * D * kStreamRows * 2 + (KV ? 2 * kStreamRows * 4 : 0));
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            tma_load_3d_hint(sm.ring[s][0][c], &tm_r0, &sm.full[s], c * 64, row, w.rplane, keep);
            tma_load_3d_hint(sm.ring[s][1][c], &tm_r1, &sm.full[s], c * 64, row, w.rplane, keep);
          }
          if constexpr (KV) {
            // the streamed queries' (lse * log2 e, D): written by the dQ pass,
            // which may still be finishing when this grid starts
            if (!dq_done) {
              asm volatile("griddepcontrol.wait;" ::: "memory");
              asm volatile("fence.proxy.async.global;" ::: "memory");  // for the TMA reads that follow
              dq_done = true;
            }
            tma_load_3d(sm.ldp[s], &tm_ldp, &sm.full[s], 2 * row, 0, w.rplane);
          }
          loads_issued = t + 1;
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
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
    // products of running tile t (ring stage t % kStages) into buffer t & 1
    auto products = [&](int t) {
      const int s = t % kStages, b = t & 1;
      const uint32_t col = kBufCol + 128u * b;
      const uint64_t r0 = d_r_k + static_cast<uint64_t>(s * kStageUnits);
      const uint64_t r1 = r0 + kSlotUnits;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t oa = (kk / 4) * (kStatSub / 16) + (kk % 4) * 2;
        const uint32_t ob = (kk / 4) * (kStreamSub / 16) + (kk % 4) * 2;
        if constexpr (KV)
          umma_bf16_ss_warp(tmem + col, d_s0 + oa, r0 + ob, id_prod, kk > 0 ? 1u : 0u);
        else  // A = Q from TMEM, 16 elements = 8 columns a step
          umma_bf16_ts_warp(tmem + col, tmem + kQCol + kk * 8, r0 + ob, id_prod, kk > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t oa = (kk / 4) * (kStatSub / 16) + (kk % 4) * 2;
        const uint32_t ob = (kk / 4) * (kStreamSub / 16) + (kk % 4) * 2;
        if constexpr (KV)
          umma_bf16_ss_warp(tmem + col + 64, d_s1 + oa, r1 + ob, id_prod, kk > 0 ? 1u : 0u);
        else  // A = dO from TMEM
          umma_bf16_ts_warp(tmem + col + 64, tmem + kQCol + D / 2 + kk * 8, r1 + ob, id_prod, kk > 0 ? 1u : 0u);
      }
      umma_commit_warp(&sm.s_full[b]);
    };
    // accumulations of running tile t; first = the unit's first tile
    auto accumulate = [&](int t, bool first) {
      const int s = t % kStages, b = t & 1;
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
    bool ok = true;
    int units = 0, tiles = 0, acc_units = 0;
    // the unit's first accumulation waits until the previous accumulators were read
    auto accumulate_unit_tile = [&](int t, bool first) -> bool {
      if (first && acc_units > 0 && !wait_all(&sm.acc_free, (acc_units - 1) & 1)) return false;
      if (!wait_all(&sm.p_full[t & 1], (t >> 1) & 1)) return false;
      tc_fence_after_sync();
      accumulate(t, first);
      return true;
    };
    for (int round = 0; ok; ++round) {
      const int u = unit_of(round);
      if (u >= n_units) break;
      const int n = work_of<KV>(u, p).count;
      // the stationary tiles in shared memory
      if (!(ok = wait_all(&sm.stat_full, units & 1))) break;
      // dQ pass: once the previous unit's products have read them, the TMEM
      // copies of Q and dO are overwritten with this unit's (A of S and dP)
      if (!KV && units > 0 && !(ok = wait_all(&sm.a_free, (units - 1) & 1))) break;
      tc_fence_after_sync();
      if constexpr (!KV) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t oa = (kk / 4) * (kStatSub / 16) + (kk % 4) * 2;
          tmem_cp_128x256b_warp(tmem + kQCol + kk * 8, d_s0 + oa);
          tmem_cp_128x256b_warp(tmem + kQCol + D / 2 + kk * 8, d_s1 + oa);
        }
        umma_commit_warp(&sm.stat_free);  // the copies have read the Q and dO tiles
        mma_issued = true;
      }
      for (int i = 0; ok && i < n; ++i) {
        const int t = tiles + i;
        if (!(ok = wait_all(&sm.full[t % kStages], (t / kStages) & 1))) break;
        tc_fence_after_sync();
        mma_issued = true;
        products(t);
        if (i == n - 1) umma_commit_warp(KV ? &sm.stat_free : &sm.a_free);  // the stationary operands' last reader
        if (i >= 1) ok = accumulate_unit_tile(t - 1, i == 1);
      }
      if (!ok) break;
      if (n == 0) {
        umma_commit_warp(KV ? &sm.stat_free : &sm.a_free);
      } else {
        if (!(ok = accumulate_unit_tile(tiles + n - 1, n == 1))) break;
        umma_commit_warp(&sm.acc_done);
        ++acc_units;
      }
      tiles += n;
      ++units;
    }
  } else if (warp == kWarpStore) {
    // ------------------------------------------------------------ dQ stores
    // dQ pass: phase 0 of dq_staged = every warp has read the first unit's
    // tiles; phase k > 0 = the dQ of the CTA's unit k - 1 is staged.  After
    // each, the stationary tiles may be reloaded: for k > 0 once the TMA
    // store of that dQ has read the staging tile.
    if (!KV && lane == 0) {
      bool ok = bwd_wait(&sm.dq_staged, 0, p, &sm.abort_flag);
      if (ok) mbar_arrive(&sm.stat_free);
      for (int round = 0; ok; ++round) {
        const int u = unit_of(round);
        if (u >= n_units) break;
        if (!(ok = bwd_wait(&sm.dq_staged, (round + 1) & 1, p, &sm.abort_flag))) break;
        const Work w = work_of<KV>(u, p);
#pragma unroll
        for (int sub = 0; sub < D / 64; ++sub) tma_store_3d(&tm_dq, sm.otile[sub], sub * 64, w.srow, w.bh);
        bulk_commit_group();
        bulk_wait_group_read0();
        mbar_arrive(&sm.stat_free);
      }
      bulk_wait_group0();  // the dQ stores have landed
    }
  } else {
    // ------------------------------------------------------------ elementwise warps
    const int quarter = warp & 3;  // TMEM lanes 32 quarter ..
    const int half = warp >> 2;    // columns 32 half .. of the 64 streamed rows
    const int r = quarter * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const long long shift = static_cast<long long>(p.Nk) - p.Nq;
    bool ok = true;
    int units = 0, tiles = 0, acc_units = 0;
    // dQ pass, once per unit and before the previous unit's epilogue: each
    // half of the warps reads its half of the columns of this thread's dO
    // and O rows (rows past Nq read as zero) and forms its share of D; the
    // two shares meet in shared memory (first half + second half, the same
    // sum in both halves) and the first half writes D for the dK/dV pass.
    // (The MMA warp copies the unit's Q and dO tiles into TMEM itself.)
    float nxt_lse = 0.f, nxt_d = 0.f;
    auto prologue = [&](int rnd, float& lse_out, float& d_out) -> bool {
      const Work wq = work_of<KV>(unit_of(rnd), p);
      const int qrow = wq.srow + r;
      const size_t l0 = static_cast<size_t>(wq.bh) * p.Nq;
      lse_out = qrow < p.Nq ? p.lse[l0 + qrow] : 0.f;  // natural log; scaled where it is used
      if (!__all_sync(0xffffffffu, bwd_wait(&sm.stat_full, rnd & 1, p, &sm.abort_flag))) return false;
      const uint8_t* dob = &sm.stat[1][0][0];
      const uint8_t* ob = &sm.otile[0][0];
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < D / 16; ++c) {
        const int cc = half * (D / 16) + c;  // 16-byte chunk of the row
        const uint32_t off = (cc >> 3) * kStatSub + (r >> 3) * 1024 + (r & 7) * 128 + (((cc & 7) ^ (r & 7)) << 4);
        float fo[8], fd[8];
        unpack_bf16x8(*reinterpret_cast<const uint4*>(ob + off), fo);
        unpack_bf16x8(*reinterpret_cast<const uint4*>(dob + off), fd);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(fd[e], fo[e], acc);
      }
      // Every warp has read the previous unit's shares once phase rnd - 1
      // of dq_staged has completed (each warp arrives there after its read).
      if (rnd > 0 && !__all_sync(0xffffffffu, bwd_wait(&sm.dq_staged, (rnd - 1) & 1, p, &sm.abort_flag))) return false;
      sm.dpart[half][r] = acc;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.dpart_full);
      if (!__all_sync(0xffffffffu, bwd_wait(&sm.dpart_full, rnd & 1, p, &sm.abort_flag))) return false;
      const float dd = sm.dpart[0][r] + sm.dpart[1][r];
      // The first unit's tiles are free (for this warp) once read; a later
      // unit's once the previous unit's dQ, staged after this read, has been
      // stored.
      __syncwarp();
      if (rnd == 0 && lane == 0) mbar_arrive(&sm.dq_staged);
      d_out = dd;
      if (half == 0 && qrow < p.Nq)
        reinterpret_cast<float2*>(p.ldp)[static_cast<size_t>(wq.bh) * p.nq_pad + qrow] = make_float2(lse_out * kLog2e, dd);
      return true;
    };
    for (int round = 0; ok; ++round) {
      const int u = unit_of(round);
      if (u >= n_units) break;
      const Work w = work_of<KV>(u, p);
      const int n = w.count;
      const int row = w.srow + r;  // key (dK/dV pass) or query row (dQ pass) of this thread
      float row_lse2 = 0.f, row_d = 0.f;
      if constexpr (!KV) {
        if (round == 0 && !(ok = prologue(0, nxt_lse, nxt_d))) break;
        row_lse2 = nxt_lse * kLog2e;
        row_d = nxt_d;
      }
      for (int i = 0; i < n; ++i) {
        const int t = tiles + i;
        const int b = t & 1;
        const int c0 = (w.first + i) * kStreamRows + half * 32;  // first streamed row of this half
        // This warp's 32 x 32 block: rows r_lo.. (keys in the dK/dV pass,
        // queries in the dQ pass), streamed columns c_lo..
        const long long r_lo = w.srow + quarter * 32, r_hi = r_lo + 31;
        const long long c_lo = c0, c_hi = c0 + 31;
        // every element visible and in range: no mask test
        const bool interior = KV ? (r_hi < p.Nk && c_hi < p.Nq && (!p.causal || r_hi <= c_lo + shift))
                                 : (r_hi < p.Nq && c_hi < p.Nk && (!p.causal || c_hi <= r_lo + shift));
        // no element visible: P and dS are zero, the products are not read
        const bool hidden = KV ? (r_lo >= p.Nk || c_lo >= p.Nq || (p.causal && r_lo > c_hi + shift))
                               : (r_lo >= p.Nq || c_lo >= p.Nk || (p.causal && c_lo > r_hi + shift));
        if (!__all_sync(0xffffffffu, bwd_wait(&sm.s_full[b], (t >> 1) & 1, p, &sm.abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t col = kBufCol + 128u * b + half * 32;
        uint32_t pk[16], dsk[16];
        if (hidden) {
#pragma unroll
          for (int c = 0; c < 16; ++c) pk[c] = dsk[c] = 0u;
        } else {
          uint32_t sv[32], dpv[32];
          tmem_ld_32x32b_x32(t_lane + col, sv);
          tmem_ld_32x32b_x32(t_lane + col + 64, dpv);
          tmem_ld_wait();
          // Visible columns of this thread's row: c in [lo, hi).  dQ pass
          // (row = query): keys below Nk and, causal, at most row + shift.
          // dK/dV pass (row = key): queries below Nq and, causal, at least
          // row - shift.  A row past the end sees nothing.
          int lo = 0, hi = 32;
          if (!interior) {
            long long l = 0, h;
            if (KV) {
              h = row < p.Nk ? static_cast<long long>(p.Nq) - c0 : 0;
              if (p.causal) l = static_cast<long long>(row) - shift - c0;
            } else {
              h = row < p.Nq ? static_cast<long long>(p.Nk) - c0 : 0;
              if (p.causal) h = min(h, static_cast<long long>(row) + shift - c0 + 1);
            }
            lo = static_cast<int>(max(0ll, min(l, 32ll)));
            hi = static_cast<int>(max(0ll, min(h, 32ll)));
          }
          // dK/dV pass: this half's 32 (lse * log2 e, D) pairs, loaded with
          // the stage's tiles (the products waited for them; so does this warp)
          const float* cols = &sm.ldp[0][0];
          if constexpr (KV) {
            const int s = t % kStages;
            if (!(ok = __all_sync(0xffffffffu, bwd_wait(&sm.full[s], (t / kStages) & 1, p, &sm.abort_flag)))) break;
            cols = &sm.ldp[s][2 * 32 * half];
          }
          if (interior)
            bwd_block<KV, false>(sv, dpv, p.scale_log2, row_lse2, row_d, cols, 0, 32, pk, dsk);
          else
            bwd_block<KV, true>(sv, dpv, p.scale_log2, row_lse2, row_d, cols, lo, hi, pk, dsk);
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
      if (!ok) break;
      if (!KV && unit_of(round + 1) < n_units && !(ok = prologue(round + 1, nxt_lse, nxt_d))) break;
      // -------------------------------------------------------- epilogue
      if (n > 0) {
        if (!(ok = __all_sync(0xffffffffu, bwd_wait(&sm.acc_done, acc_units & 1, p, &sm.abort_flag)))) break;
        tc_fence_after_sync();
      }
      {
        constexpr int kHalf = D / 2;  // accumulator columns of this thread
        const int col0 = half * kHalf;
        constexpr int n_acc = KV ? 2 : 1;
#pragma unroll 1
        for (int a = 0; a < n_acc; ++a) {
          uint32_t v[kHalf];
          if (n > 0) {
#pragma unroll
            for (int c = 0; c < kHalf / 32; ++c)
              tmem_ld_32x32b_x32(t_lane + a * D + col0 + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * c]));
            tmem_ld_wait();
            if (a == n_acc - 1) {
              // the accumulators may take the next unit's first products
              tc_fence_before_sync();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sm.acc_free);
            }
          } else {
#pragma unroll
            for (int e = 0; e < kHalf; ++e) v[e] = 0u;
          }
          // dK/dV pass: a = 0 is dV, a = 1 is dK (times scale); dQ pass: dQ (times scale)
          const float mul = (KV && a == 0) ? 1.f : p.scale;
          if constexpr (!KV) {
            // This thread's half row of dQ, in bf16, into the O tile's slot
            // where it read O (the tile's swizzled layout; rows past Nq are
            // clipped by the store), once the previous unit's dQ has left it.
            if (!(ok = __all_sync(0xffffffffu, bwd_wait(&sm.stat_free, units & 1, p, &sm.abort_flag)))) break;
            const uint32_t stage = smem_u32(&sm.otile[0][0]);
#pragma unroll
            for (int c = 0; c < kHalf / 8; ++c) {
              const int cc = half * (D / 16) + c;
              const uint32_t off = (cc >> 3) * kStatSub + (r >> 3) * 1024 + (r & 7) * 128 + (((cc & 7) ^ (r & 7)) << 4);
              st_shared_v4(stage + off,
                           pack_bf16x2(__uint_as_float(v[8 * c]) * mul, __uint_as_float(v[8 * c + 1]) * mul),
                           pack_bf16x2(__uint_as_float(v[8 * c + 2]) * mul, __uint_as_float(v[8 * c + 3]) * mul),
                           pack_bf16x2(__uint_as_float(v[8 * c + 4]) * mul, __uint_as_float(v[8 * c + 5]) * mul),
                           pack_bf16x2(__uint_as_float(v[8 * c + 6]) * mul, __uint_as_float(v[8 * c + 7]) * mul));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.dq_staged);
          } else if (row < p.Nk) {
            if (p.part == nullptr) {
              __nv_bfloat16* dst = a == 0 ? p.out1 : p.out0;
              uint4* o = reinterpret_cast<uint4*>(dst + (static_cast<size_t>(w.splane) * p.Nk + row) * D + col0);
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
              // 32-byte stores (the partials start on a 32-byte boundary)
#pragma unroll
              for (int c = 0; c < kHalf / 8; ++c)
                st_global_v8(dst + 8 * c, &v[8 * c]);
            }
          }
        }
      }
      if (!ok) break;
      if (n > 0) ++acc_units;
      tiles += n;
      ++units;
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
      if (stat_loads > 0) mbar_wait(&sm.stat_full, (stat_loads - 1) & 1, p.wait_ns);
      for (int t = loads_issued - kStages; t < loads_issued; ++t)
        if (t >= 0) mbar_wait(&sm.full[t % kStages], (t / kStages) & 1, p.wait_ns);
    }
    if (warp == kWarpMma && lane == 0 && mma_issued) {
      umma_commit(&sm.fin);
      mbar_wait(&sm.fin, 0, p.wait_ns);
    }
  }
  __syncthreads();
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
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the dK/dV pass's partials
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
  p.ldp = a.ldp;
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
  p.nq_pad = (a.Nq + 1) / 2 * 2;
  constexpr int smem_kv = static_cast<int>(bwd_smem_bytes<D, true>());
  constexpr int smem_q = static_cast<int>(bwd_smem_bytes<D, false>());
  static_assert(smem_kv <= 227 * 1024 && smem_q <= 227 * 1024, "shared memory per CTA");
  static std::atomic<int> set_kv[64] = {}, set_q[64] = {};
  cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(bwd_tc_kernel<D, true>), smem_kv, set_kv);
  if (e != cudaSuccess) return e;
  e = smem_limit_once(reinterpret_cast<const void*>(bwd_tc_kernel<D, false>), smem_q, set_q);
  if (e != cudaSuccess) return e;
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  // dQ pass first: it writes D, which the dK/dV pass reads
  if (a.Nq > 0) {
    BwdParams pq = p;
    pq.out0 = static_cast<__nv_bfloat16*>(a.dq);
    pq.out1 = nullptr;
    pq.part = nullptr;
    pq.n_tiles = (a.Nq + kStatRows - 1) / kStatRows;
    const long long units = static_cast<long long>(pq.n_tiles) * pq.n_bh;
    const long long grid = units < sms ? units : sms;
    bwd_tc_kernel<D, false><<<static_cast<unsigned>(grid), kThreads, smem_q, stream>>>(
        *a.tm_q128, *a.tm_do128, *a.tm_k64, *a.tm_v64, *a.tm_o128, *a.tm_dq128, *a.tm_ldp, pq);
  }
  const int G = a.Hq / a.Hkv;
  if (a.Nk > 0) {
    BwdParams pk = p;
    pk.out0 = static_cast<__nv_bfloat16*>(a.dk);
    pk.out1 = static_cast<__nv_bfloat16*>(a.dv);
    pk.part = G > 1 ? a.part : nullptr;
    pk.n_tiles = (a.Nk + kStatRows - 1) / kStatRows;
    const long long units = static_cast<long long>(pk.n_tiles) * pk.n_bh;
    const long long grid = units < sms ? units : sms;
    // programmatic dependent launches: each may start while the launch
    // before it finishes, and waits for it where it reads its results
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_kv;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, bwd_tc_kernel<D, true>, *a.tm_k128, *a.tm_v128, *a.tm_q64, *a.tm_do64,
                           *a.tm_k128, *a.tm_k128, *a.tm_ldp, pk);
    if (e != cudaSuccess) return e;
    if (G > 1) {
      const long long n = static_cast<long long>(a.B) * a.Hkv * a.Nk * D;
      cudaLaunchConfig_t rc = {};
      rc.gridDim = dim3(static_cast<unsigned>((n / 4 + 255) / 256));
      rc.blockDim = dim3(256);
      rc.dynamicSmemBytes = 0;
      rc.stream = stream;
      rc.attrs = pdl;
      rc.numAttrs = 1;
      const float* part = a.part;
      e = cudaLaunchKernelEx(&rc, bwd_reduce_kernel<D>, part, static_cast<__nv_bfloat16*>(a.dk),
                             static_cast<__nv_bfloat16*>(a.dv), n, G, a.scale);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, const DeviceGuard& g, cudaStream_t stream) {
  return a.d == 64 ? launch_bwd_d<64>(a, g, stream) : launch_bwd_d<128>(a, g, stream);
}

}  // namespace exattn
