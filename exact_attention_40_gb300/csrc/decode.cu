// One-token paged decode for sm_103a: split-KV partial attention plus a
// log-sum-exp merge.
//
// The key/value cache is cut into 16-token blocks; the block table maps a
// sequence's logical blocks to physical ones ("Optimizing LLM Inference
// ..." page, section Paged Attention and Dynamic KV Cache Management).  One
// (block, kv head) of K (or V) is a contiguous 16 x d bf16 span (4 KB at
// d = 128).
//
// decode_split_kernel: one CTA per (sequence, kv head, group of up to 16
//   query heads, split of SPLIT tokens).  SPLIT is kDecodeSplitTokens (512)
//   or twice that when the grid stays several waves deep with the longer
//   split (fewer CTAs, so less fixed per-CTA work per byte); the workspace
//   is laid out for 512-token splits either way.  Each of its warps
//   owns every kWarps-th block of the split and streams it through a private
//   shared-memory ring: TMA copies each span as 64-column x 16-row boxes with
//   the 128-byte swizzle, so ldmatrix reads are bank-conflict free.  Per
//   block the warp computes S = Q K^T (16 query heads x 16 tokens) and
//   O += P V with mma.sync m16n8k16 (bf16 in, fp32 accumulate; the query
//   heads of the GQA group are the 16 rows, padded with zeros), keeping an
//   online softmax (running max m, sum l) on the accumulator fragments.  At
//   the end the warps' states merge in shared memory and the split writes
//   its partial output O_s (divided by the sum of the bf16 weights P V used)
//   and lse_s (natural log, from the unrounded exponentials) to the
//   workspace.
//   When the block table cannot reach a second split (every sequence fits
//   one), the split kernel writes the final output and log-sum-exp itself
//   and the merge is not launched (it would weight the one split by 1).
// decode_combine_kernel: one CTA per (sequence, query head):
//   L = log sum_s exp(lse_s), o = sum_s exp(lse_s - L) O_s, lse = L.
//   Launched with programmatic dependent launch so its launch overlaps the
//   split kernel's tail.
#include <cuda_bf16.h>

#include "launch.h"
#include "ptx.cuh"

namespace exattn {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;
constexpr int kRows = 16;  // query heads per CTA (mma M)
constexpr int kBlk = kDecodeBlockSize;
constexpr int kMaxSplit = 2 * kDecodeSplitTokens;
static_assert((kMaxSplit / kBlk + kWarps - 1) / kWarps <= 32, "block ids are staged one per lane");
constexpr int kMergeStride = 8;  // pad of the merge staging rows (floats): conflict-free float2 stores
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr uint32_t kBoxBytes = kBlk * 64 * 2;  // 16 tokens x 64 columns, bf16

template <int D>
struct alignas(1024) DecodeSmem {
  static constexpr int kBoxes = D / 64;
  static constexpr int kStageBytes = 2 * kBoxes * kBoxBytes;  // K boxes then V boxes
  uint8_t ring[kWarps][kStages][kStageBytes];
  float wm[kWarps][kRows];  // per-warp running max (log2 units)
  float wl[kWarps][kRows];  // per-warp running sum
  float wlr[kWarps][kRows]; // per-warp running sum of the bf16-rounded weights
  uint64_t full[kWarps][kStages];
};

struct SplitParams {
  const __nv_bfloat16* q;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  float* ws_o;
  float* ws_lse;
  __nv_bfloat16* out;  // direct mode: the final output and log-sum-exp
  float* lse;
  int direct;          // every sequence fits one split: no partials, no merge
  unsigned int* status;
  unsigned long long wait_ns;
  int Hq, Hkv, group, n_chunks, num_blocks, max_blocks_per_seq, max_splits;
  float scale_log2;
};

__device__ __forceinline__ int clamp_ctx(int n, int max_ctx, unsigned int* status) {
  if (n < 0 || n > max_ctx) {
    atomicOr(status, 2u);  // EXATTN_DEVICE_BOUNDS_BIT
    n = n < 0 ? 0 : max_ctx;
  }
  return n;
}

// Shared address of the 16-byte chunk holding (token, 8 columns starting at
// col8 * 8) in a K or V tile stored as D/64 swizzled 16-row boxes.
__device__ __forceinline__ uint32_t tile_chunk(uint32_t base, int token, int col8) {
  return base + (col8 >> 3) * kBoxBytes + token * 128 + (((col8 & 7) ^ (token & 7)) << 4);
}

template <int D, int SPLIT>
__global__ void __launch_bounds__(kThreads, 2)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const SplitParams p) {
  constexpr int kKSteps = D / 16;   // QK^T k-steps
  constexpr int kNTiles = D / 8;    // P V n-tiles
  constexpr int kStageBytes = DecodeSmem<D>::kStageBytes;
  constexpr int kBoxes = DecodeSmem<D>::kBoxes;

  extern __shared__ uint8_t smem_raw[];
  DecodeSmem<D>& sm = *reinterpret_cast<DecodeSmem<D>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;  // mma group id: row g (and g + 8)
  const int t = lane & 3;   // thread in group
  const int split = blockIdx.x;
  const int hkv = blockIdx.y / p.n_chunks;
  const int chunk = blockIdx.y % p.n_chunks;
  const int seq = blockIdx.z;

  const int max_ctx = p.max_blocks_per_seq * kBlk;
  const int ctx = clamp_ctx(__ldg(p.ctx_lens + seq), max_ctx, p.status);
  const int n_splits = (ctx + SPLIT - 1) / SPLIT;
  if (split >= n_splits) {  // whole CTA: nothing of this sequence here
    if (p.direct && n_splits == 0 && split == 0) {
      // direct mode, no cached token: o = 0, lse = -inf for this CTA's heads
      const int h0 = hkv * p.group + chunk * kRows;
      const int rows = min(kRows, p.group - chunk * kRows);
      for (int idx = threadIdx.x; idx < rows * D; idx += kThreads) {
        const size_t row = static_cast<size_t>(seq) * p.Hq + h0 + idx / D;
        p.out[row * D + idx % D] = __float2bfloat16_rn(0.f);
        if (p.lse != nullptr && idx % D == 0) p.lse[row] = -INFINITY;
      }
    }
    return;
  }

  const int tok0 = split * SPLIT;
  const int tok_end = min(ctx, tok0 + SPLIT);
  const int blk0 = tok0 / kBlk;
  const int n_blk = (tok_end - tok0 + kBlk - 1) / kBlk;
  const int my_n = n_blk > warp ? (n_blk - warp + kWarps - 1) / kWarps : 0;

  // Physical block of this warp's i-th block, held by lane i.
  int phys_lane = -1;
  if (lane < my_n) {
    phys_lane = __ldg(p.block_table + static_cast<size_t>(seq) * p.max_blocks_per_seq + blk0 +
                      warp + kWarps * lane);
    if (phys_lane < 0 || phys_lane >= p.num_blocks) {
      atomicOr(p.status, 2u);
      phys_lane = -1;
    }
  }

  if (lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    for (int s = 0; s < kStages; ++s) mbar_init(&sm.full[warp][s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  const uint64_t stream_policy = l2_policy_evict_first();
  // Start the copy of this warp's i-th block into stage i % kStages (whole
  // warp calls; lane 0 issues).  A skipped block (bad table entry) still
  // completes its stage's phase so the ring stays in step.
  auto issue = [&](int i) {
    const int ph = __shfl_sync(0xffffffffu, phys_lane, i);
    if (lane == 0) {
      uint64_t* bar = &sm.full[warp][i % kStages];
      if (ph < 0) {
        mbar_arrive(bar);
      } else {
        const int row = (ph * p.Hkv + hkv) * kBlk;
        uint8_t* st = sm.ring[warp][i % kStages];
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, kStageBytes);
#pragma unroll
        for (int b = 0; b < kBoxes; ++b) {
          tma_load_3d_hint(st + b * kBoxBytes, &tm_k, bar, b * 64, row, 0, stream_policy);
          tma_load_3d_hint(st + (kBoxes + b) * kBoxBytes, &tm_v, bar, b * 64, row, 0, stream_policy);
        }
      }
    }
  };
  int issued = 0;
  for (; issued < min(my_n, kStages); ++issued) issue(issued);

  // Q as mma A fragments: row r = query head hq0 + r of this chunk (zero
  // when r >= rows_here), k-step ks covers columns 16 ks .. 16 ks + 15.
  const int hq0 = hkv * p.group + chunk * kRows;
  const int rows_here = min(kRows, p.group - chunk * kRows);
  uint32_t qa[kKSteps][4];
  {
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(p.q);
    const size_t row_lo = (static_cast<size_t>(seq) * p.Hq + hq0 + g) * (D / 2);
    const size_t row_hi = row_lo + 8 * (D / 2);
#pragma unroll
    for (int ks = 0; ks < kKSteps; ++ks) {
      const int w = ks * 8 + t;  // 32-bit word of columns 16 ks + 2t, +1
      qa[ks][0] = g < rows_here ? __ldg(q32 + row_lo + w) : 0u;
      qa[ks][1] = g + 8 < rows_here ? __ldg(q32 + row_hi + w) : 0u;
      qa[ks][2] = g < rows_here ? __ldg(q32 + row_lo + w + 4) : 0u;
      qa[ks][3] = g + 8 < rows_here ? __ldg(q32 + row_hi + w + 4) : 0u;
    }
  }

  float m[2] = {-INFINITY, -INFINITY};  // rows g, g + 8 (log2 units)
  float l[2] = {0.f, 0.f};              // this thread's partial sums of the exponentials
  float lr[2] = {0.f, 0.f};             // ... and of their bf16 roundings (what P V uses)
  float acc[kNTiles][4];
#pragma unroll
  for (int n = 0; n < kNTiles; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

  // ldmatrix lane roles: matrix mi = lane / 8, row ri = lane % 8.
  const int mi = lane >> 3, ri = lane & 7;

  for (int i = 0; i < my_n; ++i) {
    const int st = i % kStages;
    const bool waited = mbar_wait(&sm.full[warp][st], (i / kStages) & 1, p.wait_ns);
    if (!__all_sync(0xffffffffu, waited)) {
      if (lane == 0) {
        atomicOr(p.status, 1u);  // EXATTN_DEVICE_TIMEOUT_BIT
        for (int j = i + 1; j < issued; ++j)  // let copies in flight land
          mbar_wait(&sm.full[warp][j % kStages], (j / kStages) & 1, p.wait_ns);
      }
      __syncwarp();
      break;
    }
    const int ph = __shfl_sync(0xffffffffu, phys_lane, i);
    const int blk = blk0 + warp + kWarps * i;
    const int n_valid = min(kBlk, ctx - blk * kBlk);
    if (ph >= 0) {
      const uint32_t kt = smem_u32(sm.ring[warp][st]);
      const uint32_t vt = kt + kBoxes * kBoxBytes;
      // ---- S = Q K^T: two n-tiles of 8 tokens
      float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < kKSteps; ++ks) {
        uint32_t b0, b1, b2, b3;
        // matrices: (tokens 0-7, cols lo), (0-7, hi), (8-15, lo), (8-15, hi)
        ldsm_x4(tile_chunk(kt, ri + 8 * (mi >> 1), 2 * ks + (mi & 1)), b0, b1, b2, b3);
        mma_bf16_16816(c[0], qa[ks], b0, b1);
        mma_bf16_16816(c[1], qa[ks], b2, b3);
      }
      // ---- online softmax on the fragments: token of c[nt][e & 1] is
      // 8 nt + 2t + (e & 1); e < 2 is row g, e >= 2 row g + 8.
      float s[2][4];  // [row][nt * 2 + j]
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const bool ok = 8 * nt + 2 * t + jj < n_valid;
          s[0][2 * nt + jj] = ok ? c[nt][jj] * p.scale_log2 : -INFINITY;
          s[1][2 * nt + jj] = ok ? c[nt][2 + jj] * p.scale_log2 : -INFINITY;
        }
      float alpha[2];
      uint32_t pa[4];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float bm = max3f(s[r][0], s[r][1], fmaxf(s[r][2], s[r][3]));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
        const float mn = fmaxf(m[r], bm);
        alpha[r] = (mn == -INFINITY) ? 1.f : ex2_approx(m[r] - mn);
        m[r] = mn;
        float pr[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) pr[e] = (mn == -INFINITY) ? 0.f : ex2_approx(s[r][e] - mn);
        l[r] = l[r] * alpha[r] + ((pr[0] + pr[1]) + (pr[2] + pr[3]));
        pa[r] = pack_bf16x2(pr[0], pr[1]);      // a0 (row g) / a1 (row g + 8): tokens 2t, 2t+1
        pa[2 + r] = pack_bf16x2(pr[2], pr[3]);  // a2 / a3: tokens 8 + 2t, 8 + 2t + 1
        lr[r] = lr[r] * alpha[r] + ((__uint_as_float(pa[r] << 16) + __uint_as_float(pa[r] & 0xFFFF0000u)) +
                                    (__uint_as_float(pa[2 + r] << 16) + __uint_as_float(pa[2 + r] & 0xFFFF0000u)));
      }
#pragma unroll
      for (int n = 0; n < kNTiles; ++n) {
        acc[n][0] *= alpha[0];
        acc[n][1] *= alpha[0];
        acc[n][2] *= alpha[1];
        acc[n][3] *= alpha[1];
      }
      // ---- O += P V; V rows of tokens >= n_valid are zeroed in the
      // fragments (they may hold anything, NaN included).
      const bool partial = n_valid < kBlk;
      const uint32_t keep_b0 =
          (2 * t < n_valid ? 0x0000FFFFu : 0u) | (2 * t + 1 < n_valid ? 0xFFFF0000u : 0u);
      const uint32_t keep_b1 =
          (2 * t + 8 < n_valid ? 0x0000FFFFu : 0u) | (2 * t + 9 < n_valid ? 0xFFFF0000u : 0u);
#pragma unroll
      for (int n = 0; n < kNTiles; n += 2) {
        uint32_t b0, b1, b2, b3;
        // matrices: (tokens 0-7, cols n), (8-15, n), (0-7, n+1), (8-15, n+1)
        ldsm_x4_t(tile_chunk(vt, ri + 8 * (mi & 1), n + (mi >> 1)), b0, b1, b2, b3);
        if (partial) {
          b0 &= keep_b0;
          b1 &= keep_b1;
          b2 &= keep_b0;
          b3 &= keep_b1;
        }
        mma_bf16_16816(acc[n], pa, b0, b1);
        mma_bf16_16816(acc[n + 1], pa, b2, b3);
      }
    }
    __syncwarp();  // all lanes done with this stage before it is refilled
    if (issued < my_n) issue(issued++);
  }

  // ---- per-warp totals of l and l_r (the four lanes of a row group)
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
    lr[r] += __shfl_xor_sync(0xffffffffu, lr[r], 1);
    lr[r] += __shfl_xor_sync(0xffffffffu, lr[r], 2);
  }
  if (t == 0) {
    sm.wm[warp][g] = m[0];
    sm.wm[warp][g + 8] = m[1];
    sm.wl[warp][g] = l[0];
    sm.wl[warp][g + 8] = l[1];
    sm.wlr[warp][g] = lr[0];
    sm.wlr[warp][g + 8] = lr[1];
  }
  __syncthreads();  // every warp finished streaming: the rings are free
  float* wacc = reinterpret_cast<float*>(&sm.ring[0][0][0]);  // [warp][row][D]
#pragma unroll
  for (int n = 0; n < kNTiles; ++n) {
    const int col = 8 * n + 2 * t;
    *reinterpret_cast<float2*>(&wacc[(warp * kRows + g) * (D + kMergeStride) + col]) =
        make_float2(acc[n][0], acc[n][1]);
    *reinterpret_cast<float2*>(&wacc[(warp * kRows + g + 8) * (D + kMergeStride) + col]) =
        make_float2(acc[n][2], acc[n][3]);
  }
  __syncthreads();

  // ---- merge the warps; thread -> (row, column) pairs of real heads
  for (int idx = threadIdx.x; idx < rows_here * D; idx += kThreads) {
    const int r = idx / D, col = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.wm[w][r]);
    float L = 0.f, Lr = 0.f, o = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float wt = (sm.wm[w][r] == -INFINITY) ? 0.f : ex2_approx(sm.wm[w][r] - M);
        L += wt * sm.wl[w][r];
        Lr += wt * sm.wlr[w][r];
        o += wt * wacc[(w * kRows + r) * (D + kMergeStride) + col];
      }
    }
    const size_t slot = (static_cast<size_t>(seq) * p.Hq + hq0 + r) * p.max_splits + split;
    // the split's output divides by the sum of the weights P V used; its
    // log-sum-exp keeps the sum of the unrounded exponentials
    const float os = (L > 0.f) ? o / Lr : 0.f;
    const float ls = (L > 0.f) ? (M + __log2f(L)) * kLn2 : -INFINITY;
    if (p.direct) {
      // the only split: the merge would weight it by exactly 1
      const size_t row = static_cast<size_t>(seq) * p.Hq + hq0 + r;
      p.out[row * D + col] = __float2bfloat16_rn(os);
      if (p.lse != nullptr && col == 0) p.lse[row] = ls;
    } else {
      p.ws_o[slot * D + col] = os;
      if (col == 0) p.ws_lse[slot] = ls;
    }
  }
}

struct CombineParams {
  const float* ws_o;
  const float* ws_lse;
  const int32_t* ctx_lens;
  __nv_bfloat16* out;
  float* lse;
  unsigned int* status;
  int Hq, max_blocks_per_seq, max_splits;
};

template <int D, int SPLIT>
__global__ void __launch_bounds__(D) decode_combine_kernel(const CombineParams p) {
  // Programmatic dependent launch: this grid may start before the split
  // kernel has finished; wait for its results here.
  cudaGridDependencySynchronize();
  const int hq = blockIdx.x;
  const int seq = blockIdx.y;
  const int col = threadIdx.x;
  const int ctx = clamp_ctx(__ldg(p.ctx_lens + seq), p.max_blocks_per_seq * kBlk, p.status);
  const int n_splits = (ctx + SPLIT - 1) / SPLIT;
  const size_t base = (static_cast<size_t>(seq) * p.Hq + hq) * p.max_splits;
  float M = -INFINITY;
  for (int s = 0; s < n_splits; ++s) M = fmaxf(M, p.ws_lse[base + s]);
  float W = 0.f, o = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < n_splits; ++s) {
      const float ls = p.ws_lse[base + s];
      const float w = (ls == -INFINITY) ? 0.f : ex2_approx((ls - M) * kLog2e);
      W += w;
      o = fmaf(w, p.ws_o[(base + s) * D + col], o);
    }
  }
  const float res = (W > 0.f) ? o / W : 0.f;
  p.out[(static_cast<size_t>(seq) * p.Hq + hq) * D + col] = __float2bfloat16_rn(res);
  if (p.lse != nullptr && col == 0)
    p.lse[static_cast<size_t>(seq) * p.Hq + hq] = (W > 0.f) ? M + __logf(W) : -INFINITY;
}

template <int D>
size_t split_smem_bytes() {
  return sizeof(DecodeSmem<D>) + 1024;
}

template <int D, int SPLIT>
cudaError_t launch_ds(const DecodeArgs& a, const DeviceGuard& g, cudaStream_t stream) {
  static_assert(sizeof(float) * kWarps * kRows * (D + kMergeStride) <= sizeof(DecodeSmem<D>::ring),
                "merge scratch must fit in the rings");
  SplitParams sp;
  sp.q = static_cast<const __nv_bfloat16*>(a.q);
  sp.block_table = a.block_table;
  sp.ctx_lens = a.ctx_lens;
  sp.ws_o = a.ws_o;
  sp.ws_lse = a.ws_lse;
  sp.out = static_cast<__nv_bfloat16*>(a.out);
  sp.lse = a.lse;
  // Block tables too short to reach a second split: each sequence has at
  // most one, so the split kernel writes the result and no merge runs.
  sp.direct = static_cast<long long>(a.max_blocks_per_seq) * kBlk <= SPLIT ? 1 : 0;
  sp.status = g.status;
  sp.wait_ns = g.wait_ns;
  sp.Hq = a.Hq;
  sp.Hkv = a.Hkv;
  sp.group = a.Hq / a.Hkv;
  sp.n_chunks = (sp.group + kRows - 1) / kRows;
  sp.num_blocks = a.num_blocks;
  sp.max_blocks_per_seq = a.max_blocks_per_seq;
  sp.max_splits = a.max_splits;
  sp.scale_log2 = a.scale * kLog2e;
  const size_t smem = split_smem_bytes<D>();
  static std::atomic<int> smem_set[64] = {};
  cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(decode_split_kernel<D, SPLIT>),
                                  static_cast<int>(smem), smem_set);
  if (e != cudaSuccess) return e;
  dim3 grid((a.max_blocks_per_seq * kBlk + SPLIT - 1) / SPLIT, a.Hkv * sp.n_chunks, a.num_seqs);
  decode_split_kernel<D, SPLIT><<<grid, kThreads, smem, stream>>>(*a.tm_k, *a.tm_v, sp);
  e = cudaGetLastError();
  if (e != cudaSuccess || sp.direct) return e;

  CombineParams cp;
  cp.ws_o = a.ws_o;
  cp.ws_lse = a.ws_lse;
  cp.ctx_lens = a.ctx_lens;
  cp.out = static_cast<__nv_bfloat16*>(a.out);
  cp.lse = a.lse;
  cp.status = g.status;
  cp.Hq = a.Hq;
  cp.max_blocks_per_seq = a.max_blocks_per_seq;
  cp.max_splits = a.max_splits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hq, a.num_seqs);
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D, SPLIT>, cp);
}

// The longer split when even it leaves at least four waves of CTAs (two
// per SM) for the longest possible contexts.
template <int D>
cudaError_t launch_d(const DecodeArgs& a, const DeviceGuard& g, cudaStream_t stream) {
  const int sms = device_sm_count();
  const long long chunks = (a.Hq / a.Hkv + kRows - 1) / kRows;
  const long long long_splits = (static_cast<long long>(a.max_blocks_per_seq) * kBlk + kMaxSplit - 1) / kMaxSplit;
  const long long ctas = long_splits * a.num_seqs * a.Hkv * chunks;
  if (sms > 0 && ctas >= 8ll * sms) return launch_ds<D, kMaxSplit>(a, g, stream);
  return launch_ds<D, kDecodeSplitTokens>(a, g, stream);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, const DeviceGuard& g, cudaStream_t stream) {
  if (a.d == 64) return launch_d<64>(a, g, stream);
  return launch_d<128>(a, g, stream);
}

}  // namespace exattn
