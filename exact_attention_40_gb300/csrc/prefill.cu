// Prefill attention kernel for sm_103a.
//
// Computes, for every (batch, query head) and query row,
//   O = softmax(scale * Q K^T + mask) V,  lse = log sum exp(scale * Q K^T)
// streaming the keys/values of the mapped KV head in 128-row tiles, with an
// online softmax, so the score tile S and the probability tile P exist only
// in tensor memory ("Fused Kernel Compiler" page, subsection FlashAttention
// Integration, items 1-4).
//
// Persistent: one CTA per SM walks a static list of work items; an item is
// two consecutive 128-row query tiles (A, B) of one (batch, query head) that
// share every K/V tile load.  Items are numbered heaviest first and dealt in
// a snake order so heavy and light items pair up under the causal mask; the
// next item's Q copy and first S = Q K^T overlap the previous item's
// epilogue, whose O tile leaves through one TMA store.
//
// Warp roles (352 threads):
//   warps 0-3  softmax warpgroup of tile A; warps 4-7 that of tile B.  Thread
//              r of a warpgroup owns query row r of its tile, which is TMEM
//              lane r.  It reads S from TMEM, masks, keeps the running max m
//              and sums l (of the exponentials, for lse) and l_r (l plus the
//              bf16 rounding residual of each tile's largest weight, which
//              divides O), writes P (bf16) back into TMEM over S, rescales O
//              in TMEM when m grows by more than kRescaleThreshold (log2
//              units), and in the epilogue writes its lse and its O row into
//              a shared-memory staging tile.
//   warp 8     TMA producer: Q tiles through a 2-buffer ring (a tile's
//              buffer takes the next item's tile once the tile's last S has
//              been computed), K/V copies in pairs {V_(j-1), K_j} through a
//              4-slot ring; an item's last V travels with the next item's K_0.
//   warp 9     tcgen05 issuer (the whole warp runs the loop, one elected
//              lane issues), also owns the TMEM allocation.
//   warp 10    issues each staged O tile's TMA store and, once the copy has
//              read the staging tile, hands it to the warpgroup of the
//              CTA's next O tile, so no softmax warp waits for a store.
//              Issue order per key tile j:
//                S_A = Q_A K_j^T,  O_B += P_B(j-1) V_(j-1),  S_B = Q_B K_j^T,
//                O_A += P_A(j) V_j
//              so the tensor core works on one tile while the other tile's
//              softmax runs (the two warpgroups alternate).
//
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A [256,256+d),
// O_B [384,384+d).  P_X overwrites columns [0,64) of S_X as packed bf16
// pairs and is the A operand of the P*V MMA straight from TMEM.
// Shared memory: operand tiles are 128-row x 64-column bf16 sub-tiles
// (16 KB, 128-byte swizzle) exactly as TMA writes them; the MMA descriptors
// read them in place (K-major for Q and K, MN-major for V).  Every barrier
// phase is derived from running counters that carry across items.
#include <cuda_bf16.h>

#include "launch.h"
#include "ptx.cuh"

namespace exattn {
namespace {

constexpr int kBM = 128;  // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;  // keys per tile
constexpr int kThreads = 352;
constexpr int kWarpLoad = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpStore = 10;  // issues the O tiles' TMA stores
constexpr int kQBuf = 2;  // Q buffers: a tile's buffer takes the next item's tile once its last S is done
constexpr int kRing = 4;  // K/V slots: K_j in slot 2j % 4, V_j in slot (2j+1) % 4
// Copies travel in pairs: pair j = {V_(j-1), K_j} shares one completion
// barrier and one release (pair slot j % 2): K_j and V_(j-1) are both done
// once S_B(j) is issued, since O_B += P_B(j-1) V_(j-1) precedes it.
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t tmem_s_col(int x) { return x == 0 ? 0u : 128u; }
__host__ __device__ constexpr uint32_t tmem_o_col(int x) { return x == 0 ? 256u : 384u; }
constexpr float kRescaleThreshold = 8.0f;  // log2 units: p may reach 2^8 before O is rescaled
constexpr uint32_t kSubTileBytes = 128 * 64 * 2;

template <int D>
struct alignas(1024) PrefillSmem {
  uint8_t q[kQBuf][D / 64][kSubTileBytes];     // Q tiles, a ring over the CTA's tiles
  uint8_t ring[kRing][D / 64][kSubTileBytes];  // K/V tiles
  uint8_t ostage[D / 64][kSubTileBytes];       // a finished O tile, bf16, as the O tensor map stores it
  uint64_t stage_go[2];                   // warpgroup x may stage its next O tile (the previous tile's copy has read it)
  uint64_t staged;                        // the four warps of a tile's warpgroup have staged their rows
  uint64_t q_full[kQBuf], q_free[kQBuf];  // Q tile landed / Q buffer no longer read
  uint64_t full[2], empty[2];  // per pair slot: pair j = {V_(j-1), K_j}
  uint64_t s_full[2], p_full[2], o_done[2], mma_fin;
  uint32_t tmem_base;
  uint32_t abort_flag;
};

struct KernelParams {
  __nv_bfloat16* out;
  float* lse;
  unsigned int* status;
  unsigned long long wait_ns;
  int Hq, Hkv, Nq, Nk, group, n_ctiles, n_bh, n_items, causal;
  float scale_log2;  // scale * log2(e)
};

// Slow path of a bounded wait, kept out of line so that the fast path (one
// try_wait) stays short in the issue loops.  Gives up after wait_ns, or at
// once when another thread of the CTA has given up.
__device__ __noinline__ bool wait_slow(uint64_t* bar, uint32_t parity, unsigned long long wait_ns,
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

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              const KernelParams& p, uint32_t* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, p.wait_ns, p.status, abort_flag);
}

// Exponentials, packed-bf16 P and the partial row sum of one 64-key half
// (keys 64*H ..) of the score row held in sr[]; P goes to TMEM columns
// [32*H, 32*H + 32) of S.
template <int H>
__device__ __forceinline__ void softmax_exp_half(const uint32_t (&sr)[128], uint32_t t_s, float scale_log2,
                                                 float m_use, float& exact) {
  const uint64_t c2 = f2_pack(scale_log2, scale_log2);
  const uint64_t nm2 = f2_pack(-m_use, -m_use);
  uint64_t sum2[2] = {0ull, 0ull};
#pragma unroll
  for (int h = 2 * H; h < 2 * H + 2; ++h) {
    uint32_t pk[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int pair = 16 * h + c;
      const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(sr[2 * pair]), __uint_as_float(sr[2 * pair + 1])),
                                 c2, nm2);
      float x0, x1;
      f2_unpack(x2, x0, x1);
      const float p0 = ex2_approx(x0);
      const float p1 = ex2_approx(x1);
      sum2[c & 1] = f2_add(sum2[c & 1], f2_pack(p0, p1));
      pk[c] = pack_bf16x2(p0, p1);
    }
    tmem_st_32x32b_x16(t_s + 16 * h, pk);
  }
  float s0, s1;
  f2_unpack(f2_add(sum2[0], sum2[1]), s0, s1);
  exact += s0 + s1;
}

struct TileInfo {
  int n_kv;    // key tiles this query tile needs
  int n_full;  // leading key tiles that need no mask
};

__device__ __forceinline__ TileInfo tile_info(int row0, const KernelParams& p) {
  TileInfo t;
  if (row0 >= p.Nq) {
    t.n_kv = 0;
    t.n_full = 0;
    return t;
  }
  const long long shift = static_cast<long long>(p.Nk) - p.Nq;  // bottom-right alignment
  t.n_kv = (p.Nk + kBN - 1) / kBN;
  t.n_full = p.Nk / kBN;
  if (p.causal) {
    const long long last = static_cast<long long>(row0) + kBM - 1 + shift;  // last key, last row
    t.n_kv = min(t.n_kv, last < 0 ? 0 : static_cast<int>(last / kBN) + 1);
    const long long first = static_cast<long long>(row0) + shift + 1;  // keys visible to row0
    t.n_full = min(t.n_full, first <= 0 ? 0 : static_cast<int>(first / kBN));
  }
  t.n_full = min(t.n_full, t.n_kv);
  return t;
}

// One work item = two consecutive 128-row query tiles of one (batch, query
// head).  Items are numbered heaviest first (the query blocks with the most
// keys under the causal mask first, across all heads).
struct Item {
  int zq, zk, m0, n_iter;
  TileInfo ti[2];
};

__device__ __forceinline__ Item item_at(int idx, const KernelParams& p) {
  Item it;
  const int bh = idx % p.n_bh;
  const int ct = p.n_ctiles - 1 - idx / p.n_bh;
  const int hq = bh % p.Hq;
  const int b = bh / p.Hq;
  it.zq = b * p.Hq + hq;
  it.zk = b * p.Hkv + hq / p.group;
  it.m0 = ct * 2 * kBM;
  it.ti[0] = tile_info(it.m0, p);
  it.ti[1] = tile_info(it.m0 + kBM, p);
  it.n_iter = max(it.ti[0].n_kv, it.ti[1].n_kv);
  return it;
}

// Persistent schedule: CTA c takes, in round r, item r * G + c (r even) or
// r * G + G - 1 - c (r odd), G = gridDim.x.  With heaviest-first numbering
// this pairs heavy with light items.
__device__ __forceinline__ int item_index(int round) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return round * G + ((round & 1) ? (G - 1 - c) : c);
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

  if (warp == kWarpLoad && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
    mbar_init(&sm.stage_go[0], 1);
    mbar_init(&sm.stage_go[1], 1);
    mbar_init(&sm.staged, 4);
    for (int b = 0; b < kQBuf; ++b) {
      mbar_init(&sm.q_full[b], 1);
      mbar_init(&sm.q_free[b], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sm.s_full[x], 1);
      mbar_init(&sm.p_full[x], 128);
      mbar_init(&sm.o_done[x], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.mma_fin, 1);
    sm.abort_flag = 0u;
    fence_mbar_init();
  }

  int issued_pairs[2] = {0, 0};    // producer: copy pairs issued per pair slot
  int q_loads[kQBuf] = {};  // producer: Q tiles issued per buffer
  bool mma_issued = false;
  // The CTA's first copies (K_0 and Q_A of its first item: pair 0 in pair
  // slot 0, Q buffer 0) need no wait, so they go out before the TMEM
  // allocation and the set-up barrier, whose time their DRAM latency then
  // overlaps.  early_zk: that item's K/V plane (its V_0 is owed next), or -1.
  int early_zk = -1;
  if (warp == kWarpLoad && lane == 0) {
    const int idx0 = item_index(0);
    if (idx0 < p.n_items) {
      const Item it0 = item_at(idx0, p);
      if (it0.n_iter > 0 && it0.ti[0].n_kv > 0) {
        const uint64_t keep0 = l2_policy_evict_last();
        mbar_arrive_expect_tx(&sm.full[0], D * kBN * 2);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d_hint(sm.ring[0][c], &tm_k, &sm.full[0], c * 64, 0, it0.zk, keep0);
        issued_pairs[0] = 1;
        mbar_arrive_expect_tx(&sm.q_full[0], D * kBM * 2);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sm.q[0][c], &tm_q, &sm.q_full[0], c * 64, it0.m0, it0.zq);
        q_loads[0] = 1;
        early_zk = it0.zk;
      }
    }
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

  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last();  // K/V tiles are re-read by other CTAs
      const bool early = early_zk >= 0;  // pair 0 and Q_A of the first item already issued
      int g = early ? 1 : 0;    // running pair index: pair g uses pair slot g & 1
      int qt = early ? 1 : 0;   // running Q tile index: tile t uses buffer t % kQBuf
      int v_zk = early_zk, v_tile = 0;  // the V tile owed by the next pair (v_zk < 0: none)
      bool ok = true;
      // Pair g = {the owed V tile, K tile k_tile of plane k_zk (if k_zk >= 0)};
      // the V tile with the same index as that K tile is owed next, so the
      // last V of an item travels with the next item's K_0.
      auto issue_pair = [&](int k_zk, int k_tile) -> bool {
        const int ps = g & 1;
        if (g >= 2 && !wait_or_abort(&sm.empty[ps], ((g >> 1) - 1) & 1, p, &sm.abort_flag)) return false;
        const bool has_v = v_zk >= 0, has_k = k_zk >= 0;
        mbar_arrive_expect_tx(&sm.full[ps], (has_v + has_k) * D * kBN * 2);
        if (has_v) {
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d_hint(sm.ring[(2 * g + 3) % kRing][c], &tm_v, &sm.full[ps], c * 64, v_tile * kBN,
                             v_zk, keep);
        }
        if (has_k) {
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d_hint(sm.ring[(2 * g) % kRing][c], &tm_k, &sm.full[ps], c * 64, k_tile * kBN, k_zk,
                             keep);
        }
        issued_pairs[ps] = (g >> 1) + 1;
        ++g;
        v_zk = k_zk;
        v_tile = k_tile;
        return true;
      };
      for (int round = 0; ok; ++round) {
        const int idx = item_index(round);
        if (idx >= p.n_items) break;
        const Item it = item_at(idx, p);
        if (it.n_iter == 0) continue;
        // The previous item's last V is needed before this item's Q.  (The
        // first item's K_0 and Q_A went out before the set-up barrier.)
        const bool pre = round == 0 && early;
        if (!pre && !(ok = issue_pair(it.zk, 0))) break;
        for (int x = 0; x < 2; ++x) {
          if (it.ti[x].n_kv == 0) continue;
          const int b = pre && x == 0 ? 0 : qt % kQBuf;
          if (!(pre && x == 0)) {
            // the previous Q of this buffer must have been read by its last S
            if (q_loads[b] > 0 && !wait_or_abort(&sm.q_free[b], (q_loads[b] - 1) & 1, p, &sm.abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&sm.q_full[b], D * kBM * 2);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(sm.q[b][c], &tm_q, &sm.q_full[b], c * 64, it.m0 + x * kBM, it.zq);
            ++q_loads[b];
            ++qt;
          }
          if (round == 0 && x == 0) {
            // the CTA's first S needs only K_0 and Q_A: let them arrive
            // before the rest of the first item's copies share the bandwidth
            if (!(ok = wait_or_abort(&sm.full[0], 0, p, &sm.abort_flag))) break;
            if (!(ok = wait_or_abort(&sm.q_full[b], 0, p, &sm.abort_flag))) break;
          }
        }
        for (int j = 1; ok && j < it.n_iter; ++j) ok = issue_pair(it.zk, j);
      }
      if (ok && v_zk >= 0) issue_pair(-1, 0);  // the last item's last V
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop in lockstep and one elected lane
    // (always lane 0: every lane is active) issues each tcgen05 operation,
    // so descriptors and counters stay warp-uniform.
    {
      constexpr uint32_t id_qk = idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t id_pv = idesc_bf16_f32(kBM, D, false, true);
      // Descriptors are built once; a k-step, sub-tile, Q buffer or ring
      // slot moves only the start-address field (units of 16 bytes, no
      // carry: shared addresses stay below 2^18).
      constexpr uint32_t kSlotUnits = (D / 64) * kSubTileBytes / 16;
      const uint64_t dq = smem_desc(smem_u32(&sm.q[0][0][0]), 16, 1024, kSwizzle128B);
      const uint64_t dk = smem_desc(smem_u32(&sm.ring[0][0][0]), 16, 1024, kSwizzle128B);
      const uint64_t dv = smem_desc(smem_u32(&sm.ring[0][0][0]), kSubTileBytes, 1024, kSwizzle128B);
      int g = 0;                          // running pair index (as the producer's)
      int qt = 0;                         // running Q tile index (as the producer's)
      int q_waits[kQBuf] = {};            // completions of q_full[b] consumed

      // Pair g carries K_j and V_(j-1): K in ring slot (2g) % 4, V in slot
      // (2g + 3) % 4, i.e. slots 0 and 3 for even g, 2 and 1 for odd g.
      const uint64_t dk_even = dk, dk_odd = dk + 2 * kSlotUnits;
      const uint64_t dv_even = dv + 3 * kSlotUnits, dv_odd = dv + kSlotUnits;
      int p_waits0 = 0, p_waits1 = 0;  // completions of p_full[0], p_full[1] consumed

      // S_X = Q_X K^T (Q_X at descriptor qd, K at kb), then signal s_full[X]
      auto qk = [&](int x, uint64_t qd, uint64_t kb) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * (kSubTileBytes / 16) + (kk % 4) * 2;
          umma_bf16_ss_warp(tmem + tmem_s_col(x), qd + off, kb + off, id_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit_warp(&sm.s_full[x]);
      };
      // O_X (+)= P_X V with V at vb; acc0 = 0 starts O_X afresh
      auto pv = [&](int x, uint64_t vb, uint32_t acc0) {
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          umma_bf16_ts_warp(tmem + tmem_o_col(x), tmem + tmem_s_col(x) + kk * 8, vb + kk * 128, id_pv,
                            kk > 0 ? 1u : acc0);
      };
      // every lane waits; the warp goes on only if all of them saw the phase
      auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, wait_or_abort(bar, parity, p, &sm.abort_flag));
      };
      auto wait_q = [&](int qb) -> bool {
        if (!wait_all(&sm.q_full[qb], q_waits[qb] & 1)) return false;
        ++q_waits[qb];
        tc_fence_after_sync();
        return true;
      };

      bool ok = true;
      for (int round = 0; ok; ++round) {
        const int idx = item_index(round);
        if (idx >= p.n_items) break;
        const Item it = item_at(idx, p);
        if (it.n_iter == 0) continue;
        const int nA = it.ti[0].n_kv, nB = it.ti[1].n_kv, n_iter = it.n_iter;
        int qa = 0, qb = 0;  // Q buffers of tiles A and B
        if (nA > 0) qa = qt++ % kQBuf;
        if (nB > 0) qb = qt++ % kQBuf;
        const uint64_t qd_a = dq + static_cast<uint64_t>(qa * kSlotUnits);
        const uint64_t qd_b = dq + static_cast<uint64_t>(qb * kSlotUnits);
        mma_issued = true;
        // Pair base = {previous item's last V, K_0}: already complete if a
        // previous item waited for it.
        const int base = g;
        if (!wait_all(&sm.full[base & 1], (base >> 1) & 1)) break;
        tc_fence_after_sync();
        for (int j = 0; j <= n_iter; ++j) {
          const int gk = base + j;  // pair of K_j and V_(j-1)
          const bool odd = (gk & 1) != 0;
          const uint64_t kb = odd ? dk_odd : dk_even;
          const uint64_t vb_prev = odd ? dv_odd : dv_even;
          const uint64_t vb_next = odd ? dv_even : dv_odd;  // V_j, in pair gk + 1
          // ---- S_A(j) = Q_A K_j^T
          if (j < nA) {
            if (j == 0 && !(ok = wait_q(qa))) break;
            qk(0, qd_a, kb);
            if (j == nA - 1) umma_commit_warp(&sm.q_free[qa]);  // Q_A no longer read
          }
          // ---- O_B += P_B(j-1) V_(j-1)
          if (j >= 1 && j - 1 < nB) {
            if (!(ok = wait_all(&sm.p_full[1], p_waits1 & 1))) break;
            ++p_waits1;
            tc_fence_after_sync();
            pv(1, vb_prev, j == 1 ? 0u : 1u);
            if (j - 1 == nB - 1) umma_commit_warp(&sm.o_done[1]);
          }
          // Pair base + n_iter also carries the next item's K_0; that item
          // releases it after its S_B(0).
          if (j == n_iter) break;
          // ---- S_B(j) = Q_B K_j^T
          if (j < nB) {
            if (j == 0 && !(ok = wait_q(qb))) break;
            qk(1, qd_b, kb);
            if (j == nB - 1) umma_commit_warp(&sm.q_free[qb]);
          }
          umma_commit_warp(&sm.empty[gk & 1]);  // pair {V_(j-1), K_j} no longer read
          // ---- pair gk+1 = {V_j, K_(j+1)}, then O_A += P_A(j) V_j (one fence
          // after both waits)
          const int gn = gk + 1;
          if (!(ok = wait_all(&sm.full[gn & 1], (gn >> 1) & 1))) break;
          if (j < nA) {
            if (!(ok = wait_all(&sm.p_full[0], p_waits0 & 1))) break;
            ++p_waits0;
            tc_fence_after_sync();
            pv(0, vb_next, j == 0 ? 0u : 1u);
            if (j == nA - 1) umma_commit_warp(&sm.o_done[0]);
          } else {
            tc_fence_after_sync();
          }
        }
        g = base + n_iter;
      }
    }
  } else if (warp == kWarpStore) {
    // ------------------------------------------------------------ O stores
    // The CTA's O tiles in the softmax warpgroups' order (per item, A then
    // B, tiles that exist).  Before each tile but the first, the staging
    // tile (whose previous copy has been read) is handed to that tile's
    // warpgroup through the warpgroup's own barrier, so each warpgroup
    // waits for exactly its own hand-overs, in order, however many tiles
    // of the other warpgroup lie between two of its own (an item without a
    // tile B gives tile A twice in a row); then one TMA store of the tile.
    if (lane == 0) {
      int e = 0;
      bool ok = true;
      for (int round = 0; ok; ++round) {
        const int idx = item_index(round);
        if (idx >= p.n_items) break;
        const Item it = item_at(idx, p);
        for (int x = 0; x < 2 && ok; ++x) {
          const int row0 = it.m0 + x * kBM;
          if (row0 >= p.Nq) continue;
          if (e > 0) mbar_arrive(&sm.stage_go[x]);
          if (!(ok = wait_or_abort(&sm.staged, e & 1, p, &sm.abort_flag))) break;
#pragma unroll
          for (int sub = 0; sub < D / 64; ++sub) tma_store_3d(&tm_o, sm.ostage[sub], sub * 64, row0, it.zq);
          bulk_commit_group();
          bulk_wait_group_read0();
          ++e;
        }
      }
      bulk_wait_group0();  // the O stores have landed
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int x = warp >> 2;                 // 0: tile A, 1: tile B
    const int r = (warp & 3) * 32 + lane;    // row within the tile == TMEM lane
    const uint32_t t_lane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t t_s = t_lane + tmem_s_col(x);
    const uint32_t t_o = t_lane + tmem_o_col(x);
    int s_waits = 0, o_waits = 0;
    int e_base = 0;  // O tiles of this CTA's earlier items (the staging buffer's users, in order)
    int go_waits = 0;  // hand-overs of the staging tile this warpgroup has consumed
    bool ok = true;
    for (int round = 0; ok; ++round) {
      const int idx = item_index(round);
      if (idx >= p.n_items) break;
      const Item it = item_at(idx, p);
      const int row0 = it.m0 + x * kBM;
      const int e_tile = e_base + x;  // tile A is staged before tile B
      e_base += 1 + (it.m0 + kBM < p.Nq ? 1 : 0);
      if (row0 >= p.Nq) continue;  // this tile does not exist
      const int row = row0 + r;
      const int n_kv = it.ti[x].n_kv;
      const int n_full = it.ti[x].n_full;
      const long long vis_last = static_cast<long long>(row) + p.Nk - p.Nq;  // causal: keys <= vis_last
      float m_ref = -INFINITY;  // reference max, log2 units
      float l = 0.f;            // sum of the exponentials (log-sum-exp)
      float lr = 0.f;           // normaliser of O (see below)
      for (int j = 0; j < n_kv; ++j) {
        if (!__all_sync(0xffffffffu, wait_or_abort(&sm.s_full[x], s_waits & 1, p, &sm.abort_flag))) {
          ok = false;
          break;
        }
        ++s_waits;
        tc_fence_after_sync();
        uint32_t sr[kBN];
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c)
          tmem_ld_32x32b_x32(t_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
        tmem_ld_wait();

        if (j >= n_full) {
          const long long key0 = static_cast<long long>(j) * kBN;
          long long lim = static_cast<long long>(p.Nk) - key0;  // keys >= Nk do not exist
          if (p.causal) lim = min(lim, vis_last - key0 + 1);
          const int lim32 = static_cast<int>(max(-1ll, min(lim, static_cast<long long>(kBN))));
          // Keys c >= lim32 become -inf, by an explicit predicated select per
          // element (timed on a diagonal tile: ~750 cycles, against ~1,150
          // for the same mask written as a conditional store).
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            asm("{\n\t.reg .pred q;\n\tsetp.lt.s32 q, %1, %2;\n\tselp.b32 %0, %3, 0xFF800000, q;\n\t}"
                : "=r"(sr[c]) : "r"(c), "r"(lim32), "r"(sr[c]));
        }
        // Row maximum: four independent chains of three-input max.
        float acc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = fmaxf(__uint_as_float(sr[k]), __uint_as_float(sr[k + 4]));
#pragma unroll
        for (int c = 8; c < kBN; c += 8)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            acc[k] = max3f(acc[k], __uint_as_float(sr[c + k]), __uint_as_float(sr[c + 4 + k]));
        const float mxr = max3f(acc[0], acc[1], fmaxf(acc[2], acc[3]));  // raw scores
        const float mx = mxr * p.scale_log2;
        float alpha = 1.f;
        bool rescale = false;
        if (mx > m_ref + kRescaleThreshold) {
          alpha = ex2_approx(m_ref - mx);  // 0 when m_ref is -inf
          m_ref = mx;
          rescale = true;
        }
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        // p = 2^(s * scale * log2e - m); P row -> TMEM columns [0, 64) of
        // S_X (two bf16 per 32-bit column), 32 keys at a time: column 16h
        // gets keys 32h.., whose own S columns were already read.  The whole
        // row is handed over at once (two 4-MMA halves with a wait between
        // them measured slower than one 8-MMA group).
        float sum = 0.f;
        softmax_exp_half<0>(sr, t_s, p.scale_log2, m_use, sum);
        // Lazy rescale of O_X, placed after the first half so that half's
        // score registers are free.  O_X is complete up to key tile j-1
        // here: P*V_(j-1) was issued before S_X(j), and s_full fires only
        // after every earlier MMA has finished; P*V of tile j waits for the
        // hand-off below.  tcgen05.ld/st are warp-collective: the whole warp
        // rescales if any of its rows needs it (alpha is 1 for the others).
        if (j > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            uint32_t o[16];
            tmem_ld_32x32b_x16(t_o + c * 16, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st_32x32b_x16(t_o + c * 16, o);
          }
        }
        softmax_exp_half<1>(sr, t_s, p.scale_log2, m_use, sum);
        // The normaliser of O: the exact sum plus the bf16 rounding residual
        // of the tile's largest weight (computed exactly as in the loop), the
        // one weight that can dominate a row and carry its rounding error
        // into O; the log-sum-exp keeps the exact sum.
        const float pmax = ex2_approx(fmaf(mxr, p.scale_log2, -m_use));
        const uint32_t pmax_b = pack_bf16x2(pmax, 0.f);
        l = l * alpha + sum;
        lr = lr * alpha + (sum + (__uint_as_float(pmax_b << 16) - pmax));
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&sm.p_full[x]);
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      // O row -> 1/l_r -> bf16 -> the staging tile (128-byte swizzle, as
      // the O tensor map stores it), then one thread stores the whole tile
      // with TMA (rows past Nq are not written): the global writes are
      // whole lines and the warps go on at once.  The staging tile is
      // shared by the CTA's O tiles in item order, A before B.
      if (n_kv > 0) {
        if (!__all_sync(0xffffffffu, wait_or_abort(&sm.o_done[x], o_waits & 1, p, &sm.abort_flag))) break;
        ++o_waits;
        tc_fence_after_sync();
      }
      const bool row_has_keys = n_kv > 0 && l > 0.f;
      const float inv_l = row_has_keys ? 1.f / lr : 0.f;
      if (p.lse != nullptr && row < p.Nq) {
        const float lse = row_has_keys ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        p.lse[static_cast<size_t>(it.zq) * p.Nq + row] = lse;
      }
      if (e_tile > 0) {
        if (!__all_sync(0xffffffffu, wait_or_abort(&sm.stage_go[x], go_waits & 1, p, &sm.abort_flag))) break;
        ++go_waits;
      }
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (n_kv > 0) {
          tmem_ld_32x32b_x32(t_o + c * 32, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
        // columns 32c .. 32c + 31: sub-tile c / 2, 16-byte chunks 4 (c % 2) ..
        const uint32_t rb = smem_u32(&sm.ostage[c >> 1][0]) + static_cast<uint32_t>(r) * 128u;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          st_shared_v4(rb + ((static_cast<uint32_t>((c & 1) * 4 + i) ^ static_cast<uint32_t>(r & 7)) << 4),
                       w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.staged);  // this warp's rows are staged: the store warp takes it
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  const bool aborted = *reinterpret_cast<volatile uint32_t*>(&sm.abort_flag) != 0u;
  if (aborted) {
    // Drain what is still in flight before the CTA's memory goes away.
    if (warp == kWarpLoad && lane == 0) {
      for (int b = 0; b < kQBuf; ++b)
        if (q_loads[b] > 0) mbar_wait(&sm.q_full[b], (q_loads[b] - 1) & 1, p.wait_ns);
      for (int s = 0; s < 2; ++s)
        if (issued_pairs[s] > 0) mbar_wait(&sm.full[s], (issued_pairs[s] - 1) & 1, p.wait_ns);
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
  kp.out = static_cast<__nv_bfloat16*>(a.out);
  kp.lse = a.lse;
  kp.status = g.status;
  kp.wait_ns = g.wait_ns;
  kp.Hq = a.Hq;
  kp.Hkv = a.Hkv;
  kp.Nq = a.Nq;
  kp.Nk = a.Nk;
  kp.group = a.Hq / a.Hkv;
  kp.n_ctiles = (a.Nq + 2 * kBM - 1) / (2 * kBM);
  kp.n_bh = a.B * a.Hq;
  const long long n_items = static_cast<long long>(kp.n_ctiles) * kp.n_bh;
  if (n_items > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
  kp.n_items = static_cast<int>(n_items);
  kp.causal = a.causal;
  kp.scale_log2 = a.scale * 1.4426950408889634f;
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const size_t smem = smem_bytes_for<D>();
  static std::atomic<int> smem_set[64] = {};
  const cudaError_t e =
      smem_limit_once(reinterpret_cast<const void*>(prefill_kernel<D>), static_cast<int>(smem), smem_set);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (each holds all 512 TMEM columns)
  const int grid = static_cast<int>(min(n_items, static_cast<long long>(sms)));
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
