// Attention backward for sm_103a: dQ, dK, dV from dO and the forward's
// output O and log-sum-exp ("Kernel Fusion, Softmax, and Attention" page:
// training runs a different schedule of the same attention equation).  With
// P_ij = exp(s_ij - lse_i):
//   D_i   = sum_t dO_it O_it                (= sum_j P_ij dP_ij)
//   dP_ij = <dO_i, v_j>,  dS_ij = P_ij (dP_ij - D_i)
//   dV_j  = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,
//   dQ_i  = scale sum_j dS_ij k_j
// P and dS are recomputed tile by tile from Q, K and the saved LSE, never
// stored.  Three kernels, no atomics (deterministic):
//   * bwd_dsum_kernel: D per query row (one warp per row);
//   * bwd_dkdv_kernel: one CTA per 64-key block of a KV head, 4 warps x 16
//     keys; it walks every query head of the group and the query blocks the
//     mask leaves, computing S^T = K Q^T and dP^T = V dO^T, then
//     dV += P^T dO and dK += dS^T Q with P^T and dS^T turned from
//     accumulator fragments into operand fragments in registers;
//   * bwd_dq_kernel: one CTA per 64-row query block of a query head, 4 warps
//     x 16 rows; it walks the key blocks the mask leaves, recomputing S and
//     dP, and accumulates dQ += dS K.
// Tiles are 64 rows x d bf16 in shared memory, 16-byte chunks XOR-swizzled
// by row (conflict-free ldmatrix), filled by cp.async (rows past the end are
// zero) and double-buffered.  The products run on mma.sync m16n8k16 (bf16 in,
// fp32 accumulate).
#include <cuda_bf16.h>

#include "launch.h"
#include "ptx.cuh"

namespace exattn {
namespace {

constexpr int kBwdRows = 64;
constexpr int kBwdThreads = 128;

struct BwdParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const __nv_bfloat16* dout;
  const float* lse;   // [B*Hq, Nq], natural log
  const float* dsum;  // [B*Hq, Nq]: D
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* part;  // GQA: per-query-head dK, dV partials [Hq/Hkv][B*Hkv][Nk][d] each, or null
  int Hq, Hkv, Nq, Nk, causal;
  float scale, scale_log2;
};

template <int D>
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int row, int chunk) {
  return base + static_cast<uint32_t>(row * (D * 2)) + (static_cast<uint32_t>(chunk ^ (row & 7)) << 4);
}

// Rows [row0, row0 + 64) of a [n_rows, D] bf16 matrix into a swizzled tile;
// rows at or past n_rows read as zero (nothing is read for them).
template <int D>
__device__ __forceinline__ void load_tile(uint32_t sbase, const __nv_bfloat16* src, long long row0,
                                          long long n_rows) {
  constexpr int kChunks = D / 8;
  for (int e = threadIdx.x; e < kBwdRows * kChunks; e += kBwdThreads) {
    const int r = e / kChunks, c = e % kChunks;
    const bool ok = row0 + r < n_rows;
    const __nv_bfloat16* g = ok ? src + (row0 + r) * D + c * 8 : src;
    cp_async16(tile_addr<D>(sbase, r, c), g, ok);
  }
}

// A operand (16 rows x 16 k) from a row-major tile: rows r0.., k 16kk..
template <int D>
__device__ __forceinline__ void lda(uint32_t base, int r0, int kk, uint32_t (&a)[4]) {
  const int lane = threadIdx.x & 31;
  ldsm_x4(tile_addr<D>(base, r0 + (lane & 15), 2 * kk + (lane >> 4)), a[0], a[1], a[2], a[3]);
}
// B operands of two n-tiles (n0.., n0+8..) for k 16kk.. from a tile stored
// [n][k] (row n holds the k values).
template <int D>
__device__ __forceinline__ void ldb_nk(uint32_t base, int n0, int kk, uint32_t (&b)[4]) {
  const int lane = threadIdx.x & 31;
  ldsm_x4(tile_addr<D>(base, n0 + (lane & 7) + ((lane >> 4) << 3), 2 * kk + ((lane >> 3) & 1)), b[0], b[1],
          b[2], b[3]);
}
// B operands of two n-tiles (columns n0.., n0+8..) for k 16kk.. from a tile
// stored [k][n] (row k holds the n values).
template <int D>
__device__ __forceinline__ void ldb_kn(uint32_t base, int n0, int kk, uint32_t (&b)[4]) {
  const int lane = threadIdx.x & 31;
  ldsm_x4_t(tile_addr<D>(base, 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3), (n0 >> 3) + (lane >> 4)),
            b[0], b[1], b[2], b[3]);
}

// 16 x 64 fp32 accumulator fragments -> bf16 A operands for 4 k-steps of 16.
__device__ __forceinline__ void acc_to_a(const float (&c)[8][4], uint32_t (&a)[4][4]) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    a[kk][0] = pack_bf16x2(c[2 * kk][0], c[2 * kk][1]);
    a[kk][1] = pack_bf16x2(c[2 * kk][2], c[2 * kk][3]);
    a[kk][2] = pack_bf16x2(c[2 * kk + 1][0], c[2 * kk + 1][1]);
    a[kk][3] = pack_bf16x2(c[2 * kk + 1][2], c[2 * kk + 1][3]);
  }
}

// Stores a 16 x D fp32 accumulator (times mul) as bf16 rows row0.. (< n_rows).
template <int D>
__device__ __forceinline__ void store_rows(__nv_bfloat16* dst, long long row0, long long n_rows,
                                           const float (&c)[D / 8][4], float mul) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const long long row = row0 + g + 8 * h;
    if (row >= n_rows) continue;
    uint32_t* out = reinterpret_cast<uint32_t*>(dst + row * D);
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) out[nt * 4 + t] = pack_bf16x2(c[nt][2 * h] * mul, c[nt][2 * h + 1] * mul);
  }
}

// ------------------------------------------------------------------ D
template <int D>
__global__ void __launch_bounds__(256) bwd_dsum_kernel(const __nv_bfloat16* out, const __nv_bfloat16* dout,
                                                       float* dsum, long long rows) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  constexpr int kPer = D / 32;  // 2 or 4 values per lane
  const __nv_bfloat16* o = out + row * D + lane * kPer;
  const __nv_bfloat16* g = dout + row * D + lane * kPer;
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc = fmaf(__bfloat162float(o[e]), __bfloat162float(g[e]), acc);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) dsum[row] = acc;
}

// ------------------------------------------------------------------ dK, dV
// One CTA per (64-key block, query head); grid.x walks the query heads so
// that the key blocks seen by the most query rows (the first ones under the
// causal mask) are dispatched first.  With one query head per KV head the
// CTA writes dK, dV; otherwise it writes its head's fp32 partials, summed in
// head order by bwd_reduce_kernel.
template <int D>
__global__ void __launch_bounds__(kBwdThreads) bwd_dkdv_kernel(const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ float s_lse[2][kBwdRows], s_ds[2][kBwdRows];
  constexpr uint32_t kTile = kBwdRows * D * 2;
  const uint32_t base = smem_u32(smem);
  const uint32_t s_k = base, s_v = base + kTile;
  const uint32_t s_q[2] = {base + 2 * kTile, base + 4 * kTile};
  const uint32_t s_do[2] = {base + 3 * kTile, base + 5 * kTile};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int G = p.Hq / p.Hkv;
  const int bhq = blockIdx.x;             // b * Hq + hq
  const int b = bhq / p.Hq, hq = bhq % p.Hq;
  const int bk = b * p.Hkv + hq / G;      // b * Hkv + hk
  const long long n0 = static_cast<long long>(blockIdx.y) * kBwdRows;
  const long long shift = static_cast<long long>(p.Nk) - p.Nq;
  const size_t kv_off = static_cast<size_t>(bk) * p.Nk * D;
  const size_t head = static_cast<size_t>(bhq) * p.Nq;
  // query blocks that see any key of this block: rows i with n0 <= i + shift
  const int n_qb = (p.Nq + kBwdRows - 1) / kBwdRows;
  int qb_first = 0;
  if (p.causal) {
    const long long first_row = n0 - shift;
    qb_first = first_row <= 0 ? 0 : static_cast<int>(first_row / kBwdRows);
    if (qb_first > n_qb) qb_first = n_qb;
  }
  const int n_items = n_qb - qb_first;

  auto load_item = [&](int it, int buf) {
    const long long m0 = static_cast<long long>(qb_first + it) * kBwdRows;
    load_tile<D>(s_q[buf], p.q + head * D, m0, p.Nq);
    load_tile<D>(s_do[buf], p.dout + head * D, m0, p.Nq);
    if (threadIdx.x < kBwdRows) {
      const bool ok = m0 + threadIdx.x < p.Nq;
      const size_t idx = ok ? head + m0 + threadIdx.x : head;
      cp_async4(smem_u32(&s_lse[buf][threadIdx.x]), p.lse + idx, ok);
      cp_async4(smem_u32(&s_ds[buf][threadIdx.x]), p.dsum + idx, ok);
    }
  };

  load_tile<D>(s_k, p.k + kv_off, n0, p.Nk);
  load_tile<D>(s_v, p.v + kv_off, n0, p.Nk);
  if (n_items > 0) load_item(0, 0);
  cp_async_commit();

  float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[i][e] = dv[i][e] = 0.f;
  const long long key_lo = n0 + warp * 16 + g, key_hi = key_lo + 8;

  for (int it = 0; it < n_items; ++it) {
    const int buf = it & 1;
    if (it + 1 < n_items) {
      load_item(it + 1, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const long long m0 = static_cast<long long>(qb_first + it) * kBwdRows;
    // 16-query sub-blocks: S^T = K Q^T, dP^T = V dO^T for this warp's 16
    // keys, then dV += P^T dO and dK += dS^T Q.  16 rather than 32 keeps
    // S^T, dP^T and their bf16 fragments in 24 fewer registers next to the
    // 128 dK/dV accumulators.
    constexpr int kSub = 16;
    constexpr int kNT = kSub / 8, kNP = kSub / 16;
#pragma unroll 1
    for (int sub = 0; sub < kBwdRows / kSub; ++sub) {
      const int c0 = kSub * sub;
      float st[kNT][4], dpt[kNT][4];
#pragma unroll
      for (int i = 0; i < kNT; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) st[i][e] = dpt[i][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t ak[4], av[4];
        lda<D>(s_k, warp * 16, kk, ak);
        lda<D>(s_v, warp * 16, kk, av);
#pragma unroll
        for (int np = 0; np < kNP; ++np) {
          uint32_t bq[4], bd[4];
          ldb_nk<D>(s_q[buf], c0 + 16 * np, kk, bq);
          ldb_nk<D>(s_do[buf], c0 + 16 * np, kk, bd);
          mma_bf16_16816(st[2 * np], ak, bq[0], bq[1]);
          mma_bf16_16816(st[2 * np + 1], ak, bq[2], bq[3]);
          mma_bf16_16816(dpt[2 * np], av, bd[0], bd[1]);
          mma_bf16_16816(dpt[2 * np + 1], av, bd[2], bd[3]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = c0 + nt * 8 + 2 * t + (e & 1);
          const long long key = (e < 2) ? key_lo : key_hi;
          const long long qrow = m0 + col;
          const bool ok = qrow < p.Nq && key < p.Nk && (!p.causal || key <= qrow + shift);
          const float pt =
              ok ? ex2_approx(st[nt][e] * p.scale_log2 - s_lse[buf][col] * 1.4426950408889634f) : 0.f;
          st[nt][e] = pt;
          dpt[nt][e] = pt * (dpt[nt][e] - s_ds[buf][col]);
        }
      uint32_t pa[kNP][4], da[kNP][4];
#pragma unroll
      for (int kk = 0; kk < kNP; ++kk) {
        pa[kk][0] = pack_bf16x2(st[2 * kk][0], st[2 * kk][1]);
        pa[kk][1] = pack_bf16x2(st[2 * kk][2], st[2 * kk][3]);
        pa[kk][2] = pack_bf16x2(st[2 * kk + 1][0], st[2 * kk + 1][1]);
        pa[kk][3] = pack_bf16x2(st[2 * kk + 1][2], st[2 * kk + 1][3]);
        da[kk][0] = pack_bf16x2(dpt[2 * kk][0], dpt[2 * kk][1]);
        da[kk][1] = pack_bf16x2(dpt[2 * kk][2], dpt[2 * kk][3]);
        da[kk][2] = pack_bf16x2(dpt[2 * kk + 1][0], dpt[2 * kk + 1][1]);
        da[kk][3] = pack_bf16x2(dpt[2 * kk + 1][2], dpt[2 * kk + 1][3]);
      }
#pragma unroll
      for (int kk = 0; kk < kNP; ++kk)
#pragma unroll
        for (int np = 0; np < D / 16; ++np) {
          uint32_t bd[4], bq[4];
          ldb_kn<D>(s_do[buf], 16 * np, c0 / 16 + kk, bd);
          ldb_kn<D>(s_q[buf], 16 * np, c0 / 16 + kk, bq);
          mma_bf16_16816(dv[2 * np], pa[kk], bd[0], bd[1]);
          mma_bf16_16816(dv[2 * np + 1], pa[kk], bd[2], bd[3]);
          mma_bf16_16816(dk[2 * np], da[kk], bq[0], bq[1]);
          mma_bf16_16816(dk[2 * np + 1], da[kk], bq[2], bq[3]);
        }
    }
    __syncthreads();  // this buffer is refilled by the next prefetch
  }
  cp_async_wait<0>();
  if (p.part == nullptr) {
    store_rows<D>(p.dk + kv_off, n0 + warp * 16, p.Nk, dk, p.scale);
    store_rows<D>(p.dv + kv_off, n0 + warp * 16, p.Nk, dv, 1.f);
    return;
  }
  // fp32 partials of query head hq % G: [g][bk][Nk][D] for dK, then for dV
  const size_t plane = static_cast<size_t>(gridDim.x / G) * p.Nk * D;  // B*Hkv*Nk*D
  float* pk = p.part + static_cast<size_t>(hq % G) * plane + kv_off;
  float* pv = pk + static_cast<size_t>(G) * plane;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const long long row = n0 + warp * 16 + g + 8 * h;
    if (row >= p.Nk) continue;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      *reinterpret_cast<float2*>(pk + row * D + nt * 8 + 2 * t) = make_float2(dk[nt][2 * h], dk[nt][2 * h + 1]);
      *reinterpret_cast<float2*>(pv + row * D + nt * 8 + 2 * t) = make_float2(dv[nt][2 * h], dv[nt][2 * h + 1]);
    }
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

// ------------------------------------------------------------------ dQ
template <int D>
__global__ void __launch_bounds__(kBwdThreads) bwd_dq_kernel(const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr uint32_t kTile = kBwdRows * D * 2;
  const uint32_t base = smem_u32(smem);
  const uint32_t s_q = base, s_do = base + kTile;
  const uint32_t s_k[2] = {base + 2 * kTile, base + 4 * kTile};
  const uint32_t s_v[2] = {base + 3 * kTile, base + 5 * kTile};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  // grid.x walks the heads, grid.y the query blocks last to first: under
  // the causal mask the last blocks see the most keys and go first
  const int bh = blockIdx.x;
  const int b = bh / p.Hq, hq = bh % p.Hq, hk = hq / (p.Hq / p.Hkv);
  const long long m0 = static_cast<long long>(gridDim.y - 1 - blockIdx.y) * kBwdRows;
  const long long shift = static_cast<long long>(p.Nk) - p.Nq;
  const size_t q_off = static_cast<size_t>(bh) * p.Nq * D;
  const size_t kv_off = (static_cast<size_t>(b) * p.Hkv + hk) * p.Nk * D;
  int n_kb = (p.Nk + kBwdRows - 1) / kBwdRows;
  if (p.causal) {
    const long long last = m0 + kBwdRows - 1 + shift;  // last key the block's last row sees
    n_kb = last < 0 ? 0 : (last / kBwdRows + 1 < n_kb ? static_cast<int>(last / kBwdRows + 1) : n_kb);
  }
  load_tile<D>(s_q, p.q + q_off, m0, p.Nq);
  load_tile<D>(s_do, p.dout + q_off, m0, p.Nq);
  if (n_kb > 0) {
    load_tile<D>(s_k[0], p.k + kv_off, 0, p.Nk);
    load_tile<D>(s_v[0], p.v + kv_off, 0, p.Nk);
  }
  cp_async_commit();

  const long long row_lo = m0 + warp * 16 + g, row_hi = row_lo + 8;
  const size_t li = static_cast<size_t>(bh) * p.Nq;
  const float lse_lo = row_lo < p.Nq ? p.lse[li + row_lo] * 1.4426950408889634f : 0.f;
  const float lse_hi = row_hi < p.Nq ? p.lse[li + row_hi] * 1.4426950408889634f : 0.f;
  const float ds_lo = row_lo < p.Nq ? p.dsum[li + row_lo] : 0.f;
  const float ds_hi = row_hi < p.Nq ? p.dsum[li + row_hi] : 0.f;

  float dq[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dq[i][e] = 0.f;

  for (int kb = 0; kb < n_kb; ++kb) {
    const int buf = kb & 1;
    if (kb + 1 < n_kb) {
      load_tile<D>(s_k[buf ^ 1], p.k + kv_off, static_cast<long long>(kb + 1) * kBwdRows, p.Nk);
      load_tile<D>(s_v[buf ^ 1], p.v + kv_off, static_cast<long long>(kb + 1) * kBwdRows, p.Nk);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    float s[8][4], dp[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[i][e] = dp[i][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t aq[4], ad[4];
      lda<D>(s_q, warp * 16, kk, aq);
      lda<D>(s_do, warp * 16, kk, ad);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t bk_[4], bv[4];
        ldb_nk<D>(s_k[buf], 16 * np, kk, bk_);
        ldb_nk<D>(s_v[buf], 16 * np, kk, bv);
        mma_bf16_16816(s[2 * np], aq, bk_[0], bk_[1]);
        mma_bf16_16816(s[2 * np + 1], aq, bk_[2], bk_[3]);
        mma_bf16_16816(dp[2 * np], ad, bv[0], bv[1]);
        mma_bf16_16816(dp[2 * np + 1], ad, bv[2], bv[3]);
      }
    }
    const long long key0 = static_cast<long long>(kb) * kBwdRows;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const long long key = key0 + nt * 8 + 2 * t + (e & 1);
        const long long row = (e < 2) ? row_lo : row_hi;
        const bool ok = row < p.Nq && key < p.Nk && (!p.causal || key <= row + shift);
        const float pv = ok ? ex2_approx(s[nt][e] * p.scale_log2 - (e < 2 ? lse_lo : lse_hi)) : 0.f;
        s[nt][e] = pv * (dp[nt][e] - (e < 2 ? ds_lo : ds_hi));  // dS
      }
    uint32_t a[4][4];
    acc_to_a(s, a);
    // dQ += dS K (k = the 64 keys)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        uint32_t bk_[4];
        ldb_kn<D>(s_k[buf], 16 * np, kk, bk_);
        mma_bf16_16816(dq[2 * np], a[kk], bk_[0], bk_[1]);
        mma_bf16_16816(dq[2 * np + 1], a[kk], bk_[2], bk_[3]);
      }
    __syncthreads();  // this buffer is refilled by the next prefetch
  }
  cp_async_wait<0>();
  store_rows<D>(p.dq + q_off, m0 + warp * 16, p.Nq, dq, p.scale);
}

template <int D>
cudaError_t launch_bwd_d(const BwdArgs& a, cudaStream_t stream) {
  BwdParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.k = static_cast<const __nv_bfloat16*>(a.k);
  p.v = static_cast<const __nv_bfloat16*>(a.v);
  p.dout = static_cast<const __nv_bfloat16*>(a.dout);
  p.lse = a.lse;
  p.dsum = a.dsum;
  p.dq = static_cast<__nv_bfloat16*>(a.dq);
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.causal = a.causal;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  const long long rows = static_cast<long long>(a.B) * a.Hq * a.Nq;
  if (rows > 0) {
    bwd_dsum_kernel<D><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(a.out), p.dout, a.dsum, rows);
  }
  const int smem = 6 * kBwdRows * D * 2;
  static std::atomic<int> smem_dkdv[64] = {}, smem_dq[64] = {};
  cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(bwd_dkdv_kernel<D>), smem, smem_dkdv);
  if (e != cudaSuccess) return e;
  e = smem_limit_once(reinterpret_cast<const void*>(bwd_dq_kernel<D>), smem, smem_dq);
  if (e != cudaSuccess) return e;
  const int G = a.Hq / a.Hkv;
  p.part = G > 1 ? a.part : nullptr;
  if (a.Nk > 0) {
    const dim3 g_kv(a.B * a.Hq, (a.Nk + kBwdRows - 1) / kBwdRows);
    bwd_dkdv_kernel<D><<<g_kv, kBwdThreads, smem, stream>>>(p);
    if (G > 1) {
      const long long n = static_cast<long long>(a.B) * a.Hkv * a.Nk * D;
      bwd_reduce_kernel<D><<<static_cast<unsigned>((n / 4 + 255) / 256), 256, 0, stream>>>(
          a.part, p.dk, p.dv, n, G, a.scale);
    }
  }
  if (a.Nq > 0) {
    const dim3 g_q(a.B * a.Hq, (a.Nq + kBwdRows - 1) / kBwdRows);
    bwd_dq_kernel<D><<<g_q, kBwdThreads, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream) {
  return a.d == 64 ? launch_bwd_d<64>(a, stream) : launch_bwd_d<128>(a, stream);
}

}  // namespace exattn
