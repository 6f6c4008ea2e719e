// C ABI of libexattn.so (declared in include/exattn.h): argument checks,
// TMA descriptor encoding and caching, the device status word, launches.
//
// Every check runs on the host before any CUDA call, so a rejected call
// touches no GPU state.  Nothing here allocates device memory: the status
// word is a static device variable, and decode scratch is the caller's.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "../../include/exattn.h"
#include "launch.h"
#include "ptx.cuh"

namespace {

__device__ unsigned int g_status_word;  // OR of EXATTN_DEVICE_*_BIT, one per GPU

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_status_ptr[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

struct MapKey {
  uintptr_t ptr;
  int d;
  long long rows;
  long long planes;
  int box_rows;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && d == o.d && rows == o.rows && planes == o.planes &&
           box_rows == o.box_rows;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    uint64_t h = k.ptr * 0x9E3779B97F4A7C15ull;
    h ^= (static_cast<uint64_t>(k.d) << 1) + static_cast<uint64_t>(k.rows) * 0xBF58476D1CE4E5B9ull;
    h ^= static_cast<uint64_t>(k.planes) * 0x94D049BB133111EBull + static_cast<uint64_t>(k.box_rows);
    return static_cast<size_t>(h ^ (h >> 31));
  }
};
constexpr size_t kMapCacheMax = 4096;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps[kMaxDevices];

unsigned long long wait_budget_ns() {
  static const unsigned long long v = [] {
    const char* e = std::getenv("EXATTN_WAIT_TIMEOUT_NS");
    unsigned long long x = e ? std::strtoull(e, nullptr, 10) : 0ull;
    return x > 0 ? x : 2000000000ull;  // 2 s: far beyond any legitimate pipeline wait
  }();
  return v;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Current device, its status-word address and the encode entry point.
// Caller holds g_mu.
int device_state(int* dev, unsigned int** status) {
  if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return EXATTN_ERR_CUDA;
  if (g_status_ptr[*dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return EXATTN_ERR_CUDA;
    g_status_ptr[*dev] = static_cast<unsigned int*>(p);
  }
  *status = g_status_ptr[*dev];
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return EXATTN_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return EXATTN_OK;
}

// Descriptor of a bf16 tensor viewed as [planes, rows, d] (d innermost),
// loaded/stored in boxes of box_rows rows x 64 columns with 128-byte
// swizzle; rows past `rows` read as zero and are not written.  The map is
// copied to `out`, storage of the caller that outlives the launch: a later
// lookup of the same call may clear the cache when it is full.  Caller
// holds g_mu (and launches before releasing it).
int tensor_map(int dev, const void* ptr, int d, long long rows, long long planes, CUtensorMap* out,
               int box_rows = 128) {
  const MapKey key{reinterpret_cast<uintptr_t>(ptr), d, rows, planes, box_rows};
  auto& cache = g_maps[dev];
  auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return EXATTN_OK;
  }
  if (cache.size() >= kMapCacheMax) cache.clear();
  CUtensorMap m;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(rows) * d * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t elem[3] = {1, 1, 1};
  CUresult r = g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                        strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return EXATTN_ERR_CUDA;
  cache.emplace(key, m);
  *out = m;
  return EXATTN_OK;
}

// Descriptor of the backward's fp32 (lse * log2 e, D) pairs [planes][nq_pad][2]
// (nq_pad = nq rounded up to even, so rows start on 16-byte boundaries),
// viewed as [planes][1][2 nq] and loaded in boxes of 64 pairs; pairs past nq
// read as zero.  Cached and copied like tensor_map's.
int pair_map(int dev, const void* ptr, long long nq, long long planes, CUtensorMap* out) {
  const MapKey key{reinterpret_cast<uintptr_t>(ptr), 0, nq, planes, 64};  // d = 0: never a bf16 map
  auto& cache = g_maps[dev];
  auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return EXATTN_OK;
  }
  if (cache.size() >= kMapCacheMax) cache.clear();
  CUtensorMap m;
  const cuuint64_t row_bytes = static_cast<cuuint64_t>((nq + 1) / 2 * 2) * 8;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(2 * nq), 1, static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {row_bytes, row_bytes};
  cuuint32_t box[3] = {128, 1, 1};
  cuuint32_t elem[3] = {1, 1, 1};
  CUresult r = g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides,
                        box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return EXATTN_ERR_CUDA;
  cache.emplace(key, m);
  *out = m;
  return EXATTN_OK;
}

// One warp waits on a barrier with arrival count 2 that only ever sees one
// arrival, so the phase never completes and the bounded wait must expire.
__global__ void expire_wait_kernel(unsigned int* status, unsigned long long budget_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    exattn::mbar_init(&bar, 2);
    exattn::fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) exattn::mbar_arrive(&bar);
  const bool done = exattn::mbar_wait(&bar, 0, budget_ns);
  if (!__all_sync(0xffffffffu, done) && threadIdx.x == 0) atomicOr(status, EXATTN_DEVICE_TIMEOUT_BIT);
}

bool good_scale(float s) { return std::isfinite(s) && s > 0.f; }

int decode_max_splits(int max_blocks_per_seq, int block_size) {
  const long long tokens = static_cast<long long>(max_blocks_per_seq) * block_size;
  return static_cast<int>((tokens + exattn::kDecodeSplitTokens - 1) / exattn::kDecodeSplitTokens);
}

// Split-KV scratch for attn_decode_paged_static, for callers that may not
// allocate device memory.  One copy per GPU, alive until the process exits.
__device__ __align__(256) unsigned char g_static_scratch[EXATTN_STATIC_SCRATCH_BYTES];
void* g_static_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" {

const char* attn_status_string(int status) {
  switch (status) {
    case EXATTN_OK: return "EXATTN_OK";
    case EXATTN_ERR_INVALID_ARG: return "EXATTN_ERR_INVALID_ARG";
    case EXATTN_ERR_UNSUPPORTED: return "EXATTN_ERR_UNSUPPORTED";
    case EXATTN_ERR_ALIGNMENT: return "EXATTN_ERR_ALIGNMENT";
    case EXATTN_ERR_WORKSPACE: return "EXATTN_ERR_WORKSPACE";
    case EXATTN_ERR_CUDA: return "EXATTN_ERR_CUDA";
    case EXATTN_ERR_TIMEOUT: return "EXATTN_ERR_TIMEOUT";
    case EXATTN_ERR_DEVICE_BOUNDS: return "EXATTN_ERR_DEVICE_BOUNDS";
    default: return "EXATTN_UNKNOWN_STATUS";
  }
}

int attn_decode_split_tokens(void) { return exattn::kDecodeSplitTokens; }

int attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
             int Hkv, int Nq, int Nk, int d, float scale, int causal, void* stream) {
  if (B < 0 || Hq < 1 || Hkv < 1 || Nq < 0 || Nk < 0) return EXATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || !good_scale(scale)) return EXATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return EXATTN_ERR_UNSUPPORTED;
  if (Nq > (1 << 30) || Nk > (1 << 30) || B > 65535 || Hq > 65535 ||
      static_cast<long long>(B) * Hq > 0x7FFFFFFFll)
    return EXATTN_ERR_UNSUPPORTED;
  if (B == 0 || Nq == 0) return EXATTN_OK;
  if (q == nullptr || out == nullptr || (Nk > 0 && (k == nullptr || v == nullptr)))
    return EXATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || (Nk > 0 && (!aligned16(k) || !aligned16(v))) ||
      (lse != nullptr && !aligned4(lse)))
    return EXATTN_ERR_ALIGNMENT;

  exattn::PrefillArgs a;
  exattn::DeviceGuard g;
  CUtensorMap map_q, map_k, map_v, map_o;  // copied into the launch's parameters
  {
    std::lock_guard<std::mutex> lock(g_mu);
    int dev;
    int rc = device_state(&dev, &g.status);
    if (rc != EXATTN_OK) return rc;
    const long long pq = static_cast<long long>(B) * Hq, pk = static_cast<long long>(B) * Hkv;
    if ((rc = tensor_map(dev, q, d, Nq, pq, &map_q)) != EXATTN_OK) return rc;
    if ((rc = tensor_map(dev, out, d, Nq, pq, &map_o)) != EXATTN_OK) return rc;
    a.tm_q = &map_q;
    a.tm_o = &map_o;
    if (Nk > 0) {
      if ((rc = tensor_map(dev, k, d, Nk, pk, &map_k)) != EXATTN_OK) return rc;
      if ((rc = tensor_map(dev, v, d, Nk, pk, &map_v)) != EXATTN_OK) return rc;
      a.tm_k = &map_k;
      a.tm_v = &map_v;
    } else {
      a.tm_k = &map_q;  // never dereferenced: no key tiles exist
      a.tm_v = &map_q;
    }
  }
  // The lock covers only the cache lookups: the maps are this call's own
  // copies, so another thread's cache eviction cannot touch them.
  g.wait_ns = wait_budget_ns();
  a.out = out;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  if (exattn::launch_prefill(a, g, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return EXATTN_ERR_CUDA;
  return EXATTN_OK;
}

size_t attn_decode_workspace_bytes(int num_seqs, int Hq, int d, int max_blocks_per_seq,
                                   int block_size) {
  if (num_seqs < 0 || Hq < 1 || (d != 64 && d != 128) || max_blocks_per_seq < 1 ||
      block_size != exattn::kDecodeBlockSize)
    return 0;
  const size_t splits = static_cast<size_t>(decode_max_splits(max_blocks_per_seq, block_size));
  const size_t rows = static_cast<size_t>(num_seqs) * Hq * splits;
  const size_t o_bytes = rows * d * sizeof(float);
  const size_t lse_bytes = (rows * sizeof(float) + 15) & ~static_cast<size_t>(15);
  return o_bytes + lse_bytes;
}

}  // extern "C"

namespace {

// Host-side checks of attn_decode_paged's arguments (no CUDA call).
int decode_validate(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_table, const int32_t* ctx_lens, void* out, float* lse,
                    int num_seqs, int Hq, int Hkv, int d, int block_size, int num_blocks,
                    int max_blocks_per_seq, float scale, void* workspace, size_t workspace_bytes) {
  if (num_seqs < 0 || Hq < 1 || Hkv < 1 || num_blocks < 1 || max_blocks_per_seq < 1)
    return EXATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || !good_scale(scale)) return EXATTN_ERR_INVALID_ARG;
  if ((d != 64 && d != 128) || block_size != exattn::kDecodeBlockSize) return EXATTN_ERR_UNSUPPORTED;
  const int group = Hq / Hkv;
  const long long ychunks = static_cast<long long>(Hkv) * ((group + 15) / 16);
  const long long cache_rows = static_cast<long long>(num_blocks) * Hkv * block_size;
  if (num_seqs > 65535 || Hq > 65535 || ychunks > 65535 ||
      static_cast<long long>(max_blocks_per_seq) * block_size > (1 << 30) || cache_rows > 0x7FFFFFFFll)
    return EXATTN_ERR_UNSUPPORTED;
  if (num_seqs == 0) return EXATTN_OK;
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || block_table == nullptr ||
      ctx_lens == nullptr || out == nullptr)
    return EXATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      !aligned4(block_table) || !aligned4(ctx_lens) || (lse != nullptr && !aligned4(lse)))
    return EXATTN_ERR_ALIGNMENT;
  const size_t need = attn_decode_workspace_bytes(num_seqs, Hq, d, max_blocks_per_seq, block_size);
  if (workspace == nullptr || workspace_bytes < need) return EXATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return EXATTN_ERR_ALIGNMENT;
  return EXATTN_OK;
}

}  // namespace

extern "C" {

int attn_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_table, const int32_t* ctx_lens, void* out, float* lse,
                      int num_seqs, int Hq, int Hkv, int d, int block_size, int num_blocks,
                      int max_blocks_per_seq, float scale, void* workspace, size_t workspace_bytes,
                      void* stream) {
  const int vrc = decode_validate(q, k_cache, v_cache, block_table, ctx_lens, out, lse, num_seqs, Hq, Hkv,
                                  d, block_size, num_blocks, max_blocks_per_seq, scale, workspace,
                                  workspace_bytes);
  if (vrc != EXATTN_OK || num_seqs == 0) return vrc;
  const long long cache_rows = static_cast<long long>(num_blocks) * Hkv * block_size;

  exattn::DecodeArgs a;
  exattn::DeviceGuard g;
  CUtensorMap map_k, map_v;  // copied into the launch's parameters
  {
    std::lock_guard<std::mutex> lock(g_mu);
    int dev;
    int rc = device_state(&dev, &g.status);
    if (rc != EXATTN_OK) return rc;
    // Each (block, kv head) span is 16 rows of the cache viewed as
    // [num_blocks * Hkv * 16, d]; one box = 16 rows x 64 columns.
    if ((rc = tensor_map(dev, k_cache, d, cache_rows, 1, &map_k, block_size)) != EXATTN_OK) return rc;
    if ((rc = tensor_map(dev, v_cache, d, cache_rows, 1, &map_v, block_size)) != EXATTN_OK) return rc;
  }
  // The maps are this call's own copies: the launch needs no lock.
  a.tm_k = &map_k;
  a.tm_v = &map_v;
  g.wait_ns = wait_budget_ns();
  {
    const int splits = decode_max_splits(max_blocks_per_seq, block_size);
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_table = block_table;
    a.ctx_lens = ctx_lens;
    a.out = out;
    a.lse = lse;
    a.ws_o = static_cast<float*>(workspace);
    a.ws_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                        static_cast<size_t>(num_seqs) * Hq * splits * d * sizeof(float));
    a.num_seqs = num_seqs;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.num_blocks = num_blocks;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.max_splits = splits;
    a.scale = scale;
  }
  if (exattn::launch_decode(a, g, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return EXATTN_ERR_CUDA;
  return EXATTN_OK;
}

}  // extern "C"

struct exattn_graph {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

extern "C" {

int attn_decode_graph_capture(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_table, const int32_t* ctx_lens, void* out,
                              float* lse, int num_seqs, int Hq, int Hkv, int d, int block_size,
                              int num_blocks, int max_blocks_per_seq, float scale, void* workspace,
                              size_t workspace_bytes, exattn_graph** graph_out) {
  if (graph_out == nullptr) return EXATTN_ERR_INVALID_ARG;
  *graph_out = nullptr;
  if (num_seqs < 1) return EXATTN_ERR_INVALID_ARG;
  const int vrc = decode_validate(q, k_cache, v_cache, block_table, ctx_lens, out, lse, num_seqs, Hq, Hkv,
                                  d, block_size, num_blocks, max_blocks_per_seq, scale, workspace,
                                  workspace_bytes);
  if (vrc != EXATTN_OK) return vrc;
  {
    // the status word's address is looked up outside the capture
    std::lock_guard<std::mutex> lock(g_mu);
    int dev;
    unsigned int* status;
    const int rc = device_state(&dev, &status);
    if (rc != EXATTN_OK) return rc;
  }
  cudaStream_t cs;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return EXATTN_ERR_CUDA;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    cudaStreamDestroy(cs);
    return EXATTN_ERR_CUDA;
  }
  const int rc = attn_decode_paged(q, k_cache, v_cache, block_table, ctx_lens, out, lse, num_seqs, Hq,
                                   Hkv, d, block_size, num_blocks, max_blocks_per_seq, scale, workspace,
                                   workspace_bytes, cs);
  cudaGraph_t graph = nullptr;
  const cudaError_t e = cudaStreamEndCapture(cs, &graph);
  cudaStreamDestroy(cs);
  if (rc != EXATTN_OK || e != cudaSuccess) {
    if (graph != nullptr) cudaGraphDestroy(graph);
    return rc != EXATTN_OK ? rc : EXATTN_ERR_CUDA;
  }
  cudaGraphExec_t exec;
  if (cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) {
    cudaGraphDestroy(graph);
    return EXATTN_ERR_CUDA;
  }
  *graph_out = new exattn_graph{graph, exec};
  return EXATTN_OK;
}

int attn_graph_launch(exattn_graph* graph, void* stream) {
  if (graph == nullptr) return EXATTN_ERR_INVALID_ARG;
  return cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? EXATTN_OK
                                                                                          : EXATTN_ERR_CUDA;
}

int attn_graph_destroy(exattn_graph* graph) {
  if (graph == nullptr) return EXATTN_OK;
  const bool ok = cudaGraphExecDestroy(graph->exec) == cudaSuccess && cudaGraphDestroy(graph->graph) == cudaSuccess;
  delete graph;
  return ok ? EXATTN_OK : EXATTN_ERR_CUDA;
}

int attn_decode_paged_static(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_table, const int32_t* ctx_lens, void* out,
                             float* lse, int num_seqs, int Hq, int Hkv, int d, int block_size,
                             int num_blocks, int max_blocks_per_seq, float scale, void* stream) {
  // Every argument is checked on the host before any CUDA call, against a
  // stand-in for the static array (aligned, never dereferenced) of its
  // size: a request that needs more scratch fails with EXATTN_ERR_WORKSPACE.
  alignas(16) static unsigned char stand_in[16];
  const int vrc = decode_validate(q, k_cache, v_cache, block_table, ctx_lens, out, lse, num_seqs, Hq, Hkv,
                                  d, block_size, num_blocks, max_blocks_per_seq, scale, stand_in,
                                  EXATTN_STATIC_SCRATCH_BYTES);
  if (vrc != EXATTN_OK || num_seqs == 0) return vrc;
  void* scratch = nullptr;
  {
    // Once per device, with that device current: the host-side name of the
    // array is not a device address, so look the address up and keep it.
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return EXATTN_ERR_CUDA;
    if (g_static_scratch_ptr[dev] == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
        return EXATTN_ERR_CUDA;
      g_static_scratch_ptr[dev] = p;
    }
    scratch = g_static_scratch_ptr[dev];
  }
  // Same kernels as the workspace entry point.
  return attn_decode_paged(q, k_cache, v_cache, block_table, ctx_lens, out, lse, num_seqs, Hq, Hkv,
                           d, block_size, num_blocks, max_blocks_per_seq, scale, scratch,
                           EXATTN_STATIC_SCRATCH_BYTES, stream);
}

int attn_add_rms_norm(const void* x, const void* residual, const void* weight, void* out,
                      void* residual_out, int n_rows, int hidden, float eps, void* stream) {
  if (n_rows < 0 || hidden < 1 || !(eps >= 0.f) || !std::isfinite(eps)) return EXATTN_ERR_INVALID_ARG;
  if (hidden % 8 != 0 || hidden > exattn::kNormMaxHidden) return EXATTN_ERR_UNSUPPORTED;
  if (n_rows == 0) return EXATTN_OK;
  if (x == nullptr || residual == nullptr || weight == nullptr || out == nullptr || residual_out == nullptr)
    return EXATTN_ERR_INVALID_ARG;
  if (out == residual_out || out == weight || residual_out == weight) return EXATTN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(residual) || !aligned16(weight) || !aligned16(out) ||
      !aligned16(residual_out))
    return EXATTN_ERR_ALIGNMENT;
  exattn::NormArgs a;
  a.x = x;
  a.residual = residual;
  a.weight = weight;
  a.out = out;
  a.residual_out = residual_out;
  a.n_rows = n_rows;
  a.hidden = hidden;
  a.inv_hidden = 1.0f / static_cast<float>(hidden);
  a.eps = eps;
  if (exattn::launch_add_rms_norm(a, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return EXATTN_ERR_CUDA;
  return EXATTN_OK;
}

int attn_rope_cache_write(void* q, const void* k, const void* v, const int32_t* seq_ids,
                          const int32_t* positions, const int32_t* block_table, void* k_cache,
                          void* v_cache, int num_tokens, int Hq, int Hkv, int d, int num_seqs,
                          int num_blocks, int max_blocks_per_seq, float base, void* stream) {
  if (num_tokens < 0 || Hq < 1 || Hkv < 1 || num_seqs < 1 || num_blocks < 1 || max_blocks_per_seq < 1)
    return EXATTN_ERR_INVALID_ARG;
  if (!std::isfinite(base) || !(base > 1.f)) return EXATTN_ERR_INVALID_ARG;
  if (d < 16 || d > exattn::kRopeMaxDim || d % 16 != 0) return EXATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_blocks) * Hkv * 16 * d > (1ll << 40)) return EXATTN_ERR_UNSUPPORTED;
  // at most 2048 work items (8 rotated pairs or one 16-byte copy) per token
  if ((static_cast<long long>(Hq) + Hkv) * (d / 16) + static_cast<long long>(Hkv) * (d / 8) > 2048)
    return EXATTN_ERR_UNSUPPORTED;
  if (num_tokens == 0) return EXATTN_OK;
  if (q == nullptr || k == nullptr || v == nullptr || seq_ids == nullptr || positions == nullptr ||
      block_table == nullptr || k_cache == nullptr || v_cache == nullptr || k_cache == v_cache)
    return EXATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(seq_ids) & 3u) || (reinterpret_cast<uintptr_t>(positions) & 3u) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u))
    return EXATTN_ERR_ALIGNMENT;
  exattn::RopeArgs a;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    int dev;
    const int rc = device_state(&dev, &a.status);
    if (rc != EXATTN_OK) return rc;
  }
  a.q = q;
  a.k = k;
  a.v = v;
  a.seq_ids = seq_ids;
  a.positions = positions;
  a.block_table = block_table;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.num_tokens = num_tokens;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.num_seqs = num_seqs;
  a.num_blocks = num_blocks;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.log2_base = std::log2(static_cast<double>(base));
  if (exattn::launch_rope_cache_write(a, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return EXATTN_ERR_CUDA;
  return EXATTN_OK;
}

size_t attn_bwd_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d) {
  if (B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Nq < 0 || Nk < 0 || (d != 64 && d != 128)) return 0;
  // fp32 (lse * log2 e, D) pairs per query row, rows padded to an even count
  const size_t pairs = static_cast<size_t>(B) * Hq * ((static_cast<size_t>(Nq) + 1) / 2 * 2) * 2 * sizeof(float);
  // with query heads sharing a KV head: fp32 dK and dV partials per query
  // head, from a 32-byte boundary (up to 16 bytes of slack after the pairs)
  const size_t part = Hq > Hkv ? static_cast<size_t>(B) * Hq * Nk * d * sizeof(float) * 2 + 16 : 0;
  return pairs + part;
}

int attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk,
             int d, float scale, int causal, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || Hq < 1 || Hkv < 1 || Nq < 0 || Nk < 0) return EXATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || !good_scale(scale)) return EXATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return EXATTN_ERR_UNSUPPORTED;
  // 64-row blocks of either length index the second grid dimension (<= 65535)
  if (Nq > 65535 * 64 || Nk > 65535 * 64 || static_cast<long long>(B) * Hq > 65535 ||
      static_cast<long long>(B) * Hkv > 65535)
    return EXATTN_ERR_UNSUPPORTED;
  // the one-dimensional grids of the D and reduce kernels stay below 2^31
  if ((static_cast<long long>(B) * Hq * Nq + 7) / 8 > 0x7FFFFFFFll ||
      (static_cast<long long>(B) * Hkv * Nk * d / 4 + 255) / 256 > 0x7FFFFFFFll)
    return EXATTN_ERR_UNSUPPORTED;
  if (B == 0 || (Nq == 0 && Nk == 0)) return EXATTN_OK;
  // the tensors of an empty side (no queries, or no keys) may be NULL
  if ((Nq > 0 && (q == nullptr || out == nullptr || dout == nullptr || lse == nullptr || dq == nullptr)) ||
      (Nk > 0 && (k == nullptr || v == nullptr || dk == nullptr || dv == nullptr)))
    return EXATTN_ERR_INVALID_ARG;
  if ((Nq > 0 && (!aligned16(q) || !aligned16(out) || !aligned16(dout) || !aligned16(dq) || !aligned4(lse))) ||
      (Nk > 0 && (!aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv))))
    return EXATTN_ERR_ALIGNMENT;
  const size_t need = attn_bwd_workspace_bytes(B, Hq, Hkv, Nq, Nk, d);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return EXATTN_ERR_WORKSPACE;
  if (need > 0 && !aligned16(workspace)) return EXATTN_ERR_ALIGNMENT;
  exattn::BwdArgs a;
  exattn::DeviceGuard g;
  CUtensorMap maps[11];  // copied into the launches' parameters
  {
    std::lock_guard<std::mutex> lock(g_mu);
    int dev;
    int rc = device_state(&dev, &g.status);
    if (rc != EXATTN_OK) return rc;
    const long long pq = static_cast<long long>(B) * Hq, pk = static_cast<long long>(B) * Hkv;
    if (Nq > 0) {
      if ((rc = tensor_map(dev, q, d, Nq, pq, &maps[0], 64)) != EXATTN_OK) return rc;
      if ((rc = tensor_map(dev, dout, d, Nq, pq, &maps[1], 64)) != EXATTN_OK) return rc;
      if ((rc = tensor_map(dev, q, d, Nq, pq, &maps[4], 128)) != EXATTN_OK) return rc;
      if ((rc = tensor_map(dev, dout, d, Nq, pq, &maps[5], 128)) != EXATTN_OK) return rc;
      if ((rc = tensor_map(dev, out, d, Nq, pq, &maps[8], 128)) != EXATTN_OK) return rc;
      if ((rc = tensor_map(dev, dq, d, Nq, pq, &maps[9], 128)) != EXATTN_OK) return rc;
    }
    if (Nk > 0) {
      if ((rc = tensor_map(dev, k, d, Nk, pk, &maps[2], 128)) != EXATTN_OK) return rc;
      if ((rc = tensor_map(dev, v, d, Nk, pk, &maps[3], 128)) != EXATTN_OK) return rc;
      if ((rc = tensor_map(dev, k, d, Nk, pk, &maps[6], 64)) != EXATTN_OK) return rc;
      if ((rc = tensor_map(dev, v, d, Nk, pk, &maps[7], 64)) != EXATTN_OK) return rc;
    }
    // an empty side has no tiles to load: its maps are stand-ins, never used
    if (Nq > 0 && Nk > 0 && (rc = pair_map(dev, workspace, Nq, pq, &maps[10])) != EXATTN_OK) return rc;
    if (Nq == 0) maps[0] = maps[1] = maps[4] = maps[5] = maps[8] = maps[9] = maps[2];
    if (Nq == 0 || Nk == 0) maps[10] = maps[0];
    if (Nk == 0) maps[2] = maps[3] = maps[6] = maps[7] = maps[0];
  }
  g.wait_ns = wait_budget_ns();
  a.tm_q64 = &maps[0];
  a.tm_do64 = &maps[1];
  a.tm_k128 = &maps[2];
  a.tm_v128 = &maps[3];
  a.tm_q128 = &maps[4];
  a.tm_do128 = &maps[5];
  a.tm_k64 = &maps[6];
  a.tm_v64 = &maps[7];
  a.tm_o128 = &maps[8];
  a.tm_dq128 = &maps[9];
  a.tm_ldp = &maps[10];
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.dout = dout;
  a.lse = lse;
  a.ldp = static_cast<float*>(workspace);
  if (Hq > Hkv) {
    const uintptr_t p0 = reinterpret_cast<uintptr_t>(workspace) +
                         static_cast<size_t>(B) * Hq * ((static_cast<size_t>(Nq) + 1) / 2 * 2) * 2 * sizeof(float);
    a.part = reinterpret_cast<float*>((p0 + 31) & ~static_cast<uintptr_t>(31));  // 32-byte stores
  } else {
    a.part = nullptr;
  }
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  if (exattn::launch_bwd(a, g, static_cast<cudaStream_t>(stream)) != cudaSuccess) return EXATTN_ERR_CUDA;
  return EXATTN_OK;
}

int attn_get_device_status(void* stream, int* status_out) {
  if (status_out == nullptr) return EXATTN_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return EXATTN_ERR_CUDA;
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v)) != cudaSuccess) return EXATTN_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) return EXATTN_ERR_CUDA;
  *status_out = static_cast<int>(v & 0x7FFFFFFFu);
  return EXATTN_OK;
}

int attn_debug_expire_wait(unsigned long long budget_ns, void* stream) {
  if (budget_ns < 1ull || budget_ns > 10000000000ull) return EXATTN_ERR_INVALID_ARG;
  unsigned int* status = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    int dev;
    const int rc = device_state(&dev, &status);
    if (rc != EXATTN_OK) return rc;
  }
  expire_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, budget_ns);
  return cudaGetLastError() == cudaSuccess ? EXATTN_OK : EXATTN_ERR_CUDA;
}

void attn_shutdown(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (auto& m : g_maps) m.clear();
}

}  // extern "C"
