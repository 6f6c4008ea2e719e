// One-token paged decode for sm_103a: split-KV partial attention plus a
// log-sum-exp merge.
//
// The key/value cache is cut into 16-token blocks; the block table maps a
// sequence's logical blocks to physical ones ("Optimizing LLM Inference
// ..." page, section Paged Attention and Dynamic KV Cache Management).  One
// (block, kv head) of K (or V) is a contiguous 16 x d bf16 span (4 KB at
// d = 128), fetched with one bulk copy.
//
// decode_split_kernel: one CTA per (sequence, kv head, group of 4 query
//   heads, split of kDecodeSplitTokens tokens).  Each of its 4 warps owns
//   every 4th block of the split, streams it through a private 3-stage
//   shared-memory ring (cp.async.bulk + mbarrier), and keeps its own online
//   softmax state (running max m, sum l, fp32 accumulator) for the 4 query
//   heads.  At the end the 4 warp states merge in shared memory and the
//   split writes its normalised partial output O_s and lse_s (natural log)
//   to the caller's workspace.
// decode_combine_kernel: one CTA per (sequence, query head): with
//   L = log sum_s exp(lse_s), o = sum_s exp(lse_s - L) O_s, lse = L.
#include <cuda_bf16.h>

#include "launch.h"
#include "ptx.cuh"

namespace exattn {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;
constexpr int kHeads = 4;  // query heads handled per CTA (GQA group chunk)
constexpr int kBlk = kDecodeBlockSize;
constexpr int kBlocksPerSplit = kDecodeSplitTokens / kBlk;
constexpr int kMaxBlocksPerWarp = kBlocksPerSplit / kWarps;
static_assert(kBlocksPerSplit % kWarps == 0, "split must divide among warps");
static_assert(kMaxBlocksPerWarp <= 32, "block ids are staged one per lane");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

template <int D>
struct alignas(128) DecodeSmem {
  static constexpr int kTileBytes = kBlk * D * 2;
  uint8_t ring[kWarps][kStages][2][kTileBytes];  // [warp][stage][K|V]
  float p[kWarps][kBlk][kHeads];                 // probabilities of the current block
  float wm[kWarps][kHeads];                      // per-warp running max (log2 units)
  float wl[kWarps][kHeads];                      // per-warp running sum
  uint64_t full[kWarps][kStages];
};

struct SplitParams {
  const __nv_bfloat16* q;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  float* ws_o;
  float* ws_lse;
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

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int D>
__global__ void __launch_bounds__(kThreads, 2) decode_split_kernel(const SplitParams p) {
  constexpr int kTileBytes = DecodeSmem<D>::kTileBytes;
  constexpr int kLanesPerRow = D / 8;          // lanes covering one 16-byte-chunked token row
  constexpr int kTokPerInstr = 32 / kLanesPerRow;
  constexpr int kInstr = kBlk / kTokPerInstr;  // 16-byte loads per lane per K block
  constexpr int kVals = kInstr * kHeads;       // partial dot products per lane
  constexpr int kDimsPerLane = D / 32;         // P*V output columns owned per lane

  extern __shared__ uint8_t smem_raw[];
  DecodeSmem<D>& sm = *reinterpret_cast<DecodeSmem<D>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int hkv = blockIdx.y / p.n_chunks;
  const int chunk = blockIdx.y % p.n_chunks;
  const int seq = blockIdx.z;

  const int max_ctx = p.max_blocks_per_seq * kBlk;
  const int ctx = clamp_ctx(__ldg(p.ctx_lens + seq), max_ctx, p.status);
  const int n_splits = (ctx + kDecodeSplitTokens - 1) / kDecodeSplitTokens;
  if (split >= n_splits) return;  // whole CTA: nothing of this sequence here

  const int tok0 = split * kDecodeSplitTokens;
  const int tok_end = min(ctx, tok0 + kDecodeSplitTokens);
  const int blk0 = tok0 / kBlk;
  const int n_blk = (tok_end - tok0 + kBlk - 1) / kBlk;
  // this warp's blocks: blk0 + warp + kWarps * i
  const int my_n = n_blk > warp ? (n_blk - warp + kWarps - 1) / kWarps : 0;

  // Physical block ids of this warp's blocks, one per lane.
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
    for (int s = 0; s < kStages; ++s) mbar_init(&sm.full[warp][s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  const size_t head_stride = static_cast<size_t>(kTileBytes);                 // (block, head) span
  const size_t block_stride = static_cast<size_t>(p.Hkv) * kTileBytes;      // one physical block
  const uint64_t stream_policy = l2_policy_evict_first();

  // Query rows of the 4 heads, restricted to this lane's 8 dims, in fp32.
  const int hq0 = hkv * p.group + chunk * kHeads;
  const int dim0 = 8 * (lane % kLanesPerRow);
  float qv[kHeads][8];
#pragma unroll
  for (int h = 0; h < kHeads; ++h) {
    const bool valid = chunk * kHeads + h < p.group;
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (valid)
      raw = *reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(seq) * p.Hq + hq0 + h) * D + dim0);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      qv[h][2 * e] = bf16lo(w[e]);
      qv[h][2 * e + 1] = bf16hi(w[e]);
    }
  }

  float m[kHeads], lpart[2], acc[kHeads][kDimsPerLane];
#pragma unroll
  for (int h = 0; h < kHeads; ++h) {
    m[h] = -INFINITY;
#pragma unroll
    for (int e = 0; e < kDimsPerLane; ++e) acc[h][e] = 0.f;
  }
  lpart[0] = lpart[1] = 0.f;

  // Start the copy of this warp's i-th block into stage i % kStages (the
  // whole warp calls this; lane 0 issues).  A skipped block (bad table
  // entry) still completes its stage's phase so the ring stays in step.
  auto issue = [&](int i) {
    const int ph = __shfl_sync(0xffffffffu, phys_lane, i);
    if (lane == 0) {
      uint64_t* bar = &sm.full[warp][i % kStages];
      if (ph < 0) {
        mbar_arrive(bar);
      } else {
        const size_t off = static_cast<size_t>(ph) * block_stride + hkv * head_stride;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, 2 * kTileBytes);
        bulk_load_hint(sm.ring[warp][i % kStages][0], p.k_cache + off, kTileBytes, bar, stream_policy);
        bulk_load_hint(sm.ring[warp][i % kStages][1], p.v_cache + off, kTileBytes, bar, stream_policy);
      }
    }
  };
  int issued = 0;
  for (; issued < min(my_n, kStages); ++issued) issue(issued);

  const int my_h0 = 2 * (lane & 1);  // heads whose scores this lane holds after the reduction
  for (int i = 0; i < my_n; ++i) {
    const int st = i % kStages;
    const bool waited = mbar_wait(&sm.full[warp][st], (i / kStages) & 1, p.wait_ns);
    if (!__all_sync(0xffffffffu, waited)) {
      if (lane == 0) {
        atomicOr(p.status, 1u);  // EXATTN_DEVICE_TIMEOUT_BIT
        // let copies still in flight land before the ring is reused
        for (int j = i + 1; j < issued; ++j)
          mbar_wait(&sm.full[warp][j % kStages], (j / kStages) & 1, p.wait_ns);
      }
      __syncwarp();
      break;
    }
    const int ph = __shfl_sync(0xffffffffu, phys_lane, i);
    const int blk = blk0 + warp + kWarps * i;
    const int n_valid = min(kBlk, ctx - blk * kBlk);
    if (ph >= 0) {
      const uint8_t* kt = sm.ring[warp][st][0];
      const uint8_t* vt = sm.ring[warp][st][1];
      // ---- scores: lane reads 16 bytes of token (kTokPerInstr*t + lane/kLanesPerRow)
      float part[kVals];
#pragma unroll
      for (int t = 0; t < kInstr; ++t) {
        const uint4 kw = *reinterpret_cast<const uint4*>(kt + t * 512 + lane * 16);
        const uint32_t w[4] = {kw.x, kw.y, kw.z, kw.w};
        float kf[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          kf[2 * e] = bf16lo(w[e]);
          kf[2 * e + 1] = bf16hi(w[e]);
        }
#pragma unroll
        for (int h = 0; h < kHeads; ++h) {
          float a = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) a = fmaf(qv[h][e], kf[e], a);
          part[t * kHeads + h] = a;
        }
      }
      // ---- reduce-scatter across the kLanesPerRow lanes sharing a token:
      // afterwards lane holds values 2*(lane % kLanesPerRow) + {0,1}.
      int cnt = kVals;
#pragma unroll
      for (int mask = kLanesPerRow / 2; mask >= 1; mask >>= 1) {
        const int half = cnt / 2;
        const bool upper = (lane & mask) != 0;
#pragma unroll
        for (int k = 0; k < kVals / 2; ++k) {
          if (k < half) {
            const float send = upper ? part[k] : part[k + half];
            const float keep = upper ? part[k + half] : part[k];
            part[k] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
          }
        }
        cnt = half;
      }
      // value index v = 2*(lane % kLanesPerRow) + e  ->  instr t = v / 4, head v % 4
      const int tok = kTokPerInstr * ((lane % kLanesPerRow) >> 1) + lane / kLanesPerRow;
      float sc[2];
#pragma unroll
      for (int e = 0; e < 2; ++e)
        sc[e] = (tok < n_valid) ? part[e] * p.scale_log2 : -INFINITY;
      // ---- block max per head (lanes with equal lane&1 hold the same heads)
      float bm[2] = {sc[0], sc[1]};
#pragma unroll
      for (int mask = 2; mask <= 16; mask <<= 1) {
        bm[0] = fmaxf(bm[0], __shfl_xor_sync(0xffffffffu, bm[0], mask));
        bm[1] = fmaxf(bm[1], __shfl_xor_sync(0xffffffffu, bm[1], mask));
      }
      const float om0 = __shfl_xor_sync(0xffffffffu, bm[0], 1);
      const float om1 = __shfl_xor_sync(0xffffffffu, bm[1], 1);
      const bool odd = (lane & 1) != 0;  // this lane holds heads 2,3 (else 0,1)
      float blkmax[kHeads];
      blkmax[0] = odd ? om0 : bm[0];
      blkmax[1] = odd ? om1 : bm[1];
      blkmax[2] = odd ? bm[0] : om0;
      blkmax[3] = odd ? bm[1] : om1;
      float alpha[kHeads];
#pragma unroll
      for (int h = 0; h < kHeads; ++h) {
        const float mn = fmaxf(m[h], blkmax[h]);
        alpha[h] = (mn == -INFINITY) ? 1.f : ex2_approx(m[h] - mn);
        m[h] = mn;
      }
      float pv[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float mh = odd ? m[2 + e] : m[e];
        const float ah = odd ? alpha[2 + e] : alpha[e];
        pv[e] = (mh == -INFINITY) ? 0.f : ex2_approx(sc[e] - mh);
        lpart[e] = lpart[e] * ah + pv[e];
      }
      *reinterpret_cast<float2*>(&sm.p[warp][tok][my_h0]) = make_float2(pv[0], pv[1]);
      __syncwarp();
      // ---- O += P V over the valid tokens; lane owns columns [kDimsPerLane*lane, +kDimsPerLane)
#pragma unroll
      for (int h = 0; h < kHeads; ++h)
#pragma unroll
        for (int e = 0; e < kDimsPerLane; ++e) acc[h][e] *= alpha[h];
      for (int t = 0; t < n_valid; ++t) {
        const float4 pt = *reinterpret_cast<const float4*>(&sm.p[warp][t][0]);
        float vf[kDimsPerLane];
        if constexpr (kDimsPerLane == 4) {
          const uint2 vw = *reinterpret_cast<const uint2*>(vt + t * (D * 2) + lane * 8);
          vf[0] = bf16lo(vw.x);
          vf[1] = bf16hi(vw.x);
          vf[2] = bf16lo(vw.y);
          vf[3] = bf16hi(vw.y);
        } else {
          const uint32_t vw = *reinterpret_cast<const uint32_t*>(vt + t * (D * 2) + lane * 4);
          vf[0] = bf16lo(vw);
          vf[1] = bf16hi(vw);
        }
        const float pp[kHeads] = {pt.x, pt.y, pt.z, pt.w};
#pragma unroll
        for (int h = 0; h < kHeads; ++h)
#pragma unroll
          for (int e = 0; e < kDimsPerLane; ++e) acc[h][e] = fmaf(pp[h], vf[e], acc[h][e]);
      }
    }
    __syncwarp();  // all lanes done with this stage before it is refilled
    if (issued < my_n) issue(issued++);
  }

  // ---- per-warp totals of l for all 4 heads
#pragma unroll
  for (int mask = 2; mask <= 16; mask <<= 1) {
    lpart[0] += __shfl_xor_sync(0xffffffffu, lpart[0], mask);
    lpart[1] += __shfl_xor_sync(0xffffffffu, lpart[1], mask);
  }
  if (lane < 2) {
    sm.wm[warp][2 * lane] = m[2 * lane];
    sm.wm[warp][2 * lane + 1] = m[2 * lane + 1];
    sm.wl[warp][2 * lane] = lpart[0];
    sm.wl[warp][2 * lane + 1] = lpart[1];
  }
  __syncthreads();  // every warp finished streaming: the rings are free
  float* wacc = reinterpret_cast<float*>(&sm.ring[0][0][0][0]);  // [warp][head][D]
#pragma unroll
  for (int h = 0; h < kHeads; ++h)
#pragma unroll
    for (int e = 0; e < kDimsPerLane; ++e)
      wacc[(warp * kHeads + h) * D + kDimsPerLane * lane + e] = acc[h][e];
  __syncthreads();

  // ---- merge the 4 warps; thread -> (head, column) pairs
  for (int idx = threadIdx.x; idx < kHeads * D; idx += kThreads) {
    const int h = idx / D, col = idx % D;
    if (chunk * kHeads + h >= p.group) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.wm[w][h]);
    float L = 0.f, o = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float wt = (sm.wm[w][h] == -INFINITY) ? 0.f : ex2_approx(sm.wm[w][h] - M);
        L += wt * sm.wl[w][h];
        o += wt * wacc[(w * kHeads + h) * D + col];
      }
    }
    const int hq = hq0 + h;
    const size_t slot = (static_cast<size_t>(seq) * p.Hq + hq) * p.max_splits + split;
    p.ws_o[slot * D + col] = (L > 0.f) ? o / L : 0.f;
    if (col == 0) p.ws_lse[slot] = (L > 0.f) ? (M + __log2f(L)) * kLn2 : -INFINITY;
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

template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const CombineParams p) {
  const int hq = blockIdx.x;
  const int seq = blockIdx.y;
  const int col = threadIdx.x;
  const int ctx = clamp_ctx(__ldg(p.ctx_lens + seq), p.max_blocks_per_seq * kBlk, p.status);
  const int n_splits = (ctx + kDecodeSplitTokens - 1) / kDecodeSplitTokens;
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
  return sizeof(DecodeSmem<D>) + 128;
}

template <int D>
cudaError_t launch_d(const DecodeArgs& a, const DeviceGuard& g, cudaStream_t stream) {
  static_assert(sizeof(float) * kWarps * kHeads * D <= sizeof(DecodeSmem<D>::ring),
                "merge scratch must fit in the rings");
  SplitParams sp;
  sp.q = static_cast<const __nv_bfloat16*>(a.q);
  sp.k_cache = static_cast<const uint8_t*>(a.k_cache);
  sp.v_cache = static_cast<const uint8_t*>(a.v_cache);
  sp.block_table = a.block_table;
  sp.ctx_lens = a.ctx_lens;
  sp.ws_o = a.ws_o;
  sp.ws_lse = a.ws_lse;
  sp.status = g.status;
  sp.wait_ns = g.wait_ns;
  sp.Hq = a.Hq;
  sp.Hkv = a.Hkv;
  sp.group = a.Hq / a.Hkv;
  sp.n_chunks = (sp.group + kHeads - 1) / kHeads;
  sp.num_blocks = a.num_blocks;
  sp.max_blocks_per_seq = a.max_blocks_per_seq;
  sp.max_splits = a.max_splits;
  sp.scale_log2 = a.scale * kLog2e;
  const size_t smem = split_smem_bytes<D>();
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(a.max_splits, a.Hkv * sp.n_chunks, a.num_seqs);
  decode_split_kernel<D><<<grid, kThreads, smem, stream>>>(sp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

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
  decode_combine_kernel<D><<<dim3(a.Hq, a.num_seqs), D, 0, stream>>>(cp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, const DeviceGuard& g, cudaStream_t stream) {
  if (a.d == 64) return launch_d<64>(a, g, stream);
  return launch_d<128>(a, g, stream);
}

}  // namespace exattn
