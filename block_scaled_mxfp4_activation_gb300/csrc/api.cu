// The C ABI: argument checks, device checks, tensor-map encoding, plan choice
// and launches.  Nothing here allocates device memory.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "internal.h"

namespace mxfp4 {
namespace {

std::atomic<uint64_t> g_timeout_ns{1000000000ull};
std::atomic<int> g_programmatic{3};

// The CUDA error behind the last MXFP4_ERR_CUDA status of this thread.
thread_local char g_last_error[256] = "";

mxfp4_status_t cuda_failure(const char* what, cudaError_t e) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
  return MXFP4_ERR_CUDA;
}

mxfp4_status_t failure(const char* what) {
  snprintf(g_last_error, sizeof(g_last_error), "%s", what);
  return MXFP4_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The device's address of pinned, mapped host memory (null for anything else:
// pageable or device memory, or a pointer CUDA does not know).
const void* device_view(const void* host_ptr) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, host_ptr) != cudaSuccess) {
    cudaGetLastError();  // not a CUDA error the caller should see
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

struct DeviceInfo {
  bool ok = false;
  cudaDeviceProp prop{};
};

// Properties of the current device, cached per device; ok only on sm_103.
const DeviceInfo* current_device(mxfp4_status_t* st) {
  static DeviceInfo info[64];
  static std::once_flag once[64];
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    *st = e != cudaSuccess ? cuda_failure("cudaGetDevice", e) : failure("device index out of range");
    return nullptr;
  }
  std::call_once(once[dev], [dev]() {
    if (cudaGetDeviceProperties(&info[dev].prop, dev) == cudaSuccess)
      info[dev].ok = info[dev].prop.major == 10 && info[dev].prop.minor == 3;
  });
  if (!info[dev].ok) {
    *st = MXFP4_ERR_UNSUPPORTED_DEVICE;
    return nullptr;
  }
  *st = MXFP4_OK;
  return &info[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Encodes a 2-D tiled tensor map (element strides 1, no interleave, L2
// promotion 256 B, no OOB fill), reusing the result of an identical earlier
// request from this thread: a map holds only the address, shape, strides and
// box, so repeated calls on the same buffers (every layer call, every step of
// a loop) skip the encoder.  A direct-mapped cache per thread: one hashed slot
// per request, so a lookup is one comparison whether it hits or misses.
bool encode_2d(CUtensorMapDataType type, const void* base, uint64_t dim0, uint64_t dim1, uint64_t stride1,
               uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle, CUtensorMap* map) {
  struct Entry {
    const void* base;
    uint64_t dim0, dim1, stride1;
    uint32_t box0, box1;
    int type, swizzle;
    bool valid;
    CUtensorMap map;
  };
  constexpr int kSlots = 256;
  thread_local Entry cache[kSlots] = {};
  uint64_t h = reinterpret_cast<uintptr_t>(base) * 0x9E3779B97F4A7C15ull;
  h ^= (dim0 * 0xC2B2AE3D27D4EB4Full) ^ (dim1 * 0x165667B19E3779F9ull) ^ (stride1 << 7) ^
       (static_cast<uint64_t>(box0) << 17) ^ (static_cast<uint64_t>(box1) << 29) ^
       (static_cast<uint64_t>(type) << 41) ^ (static_cast<uint64_t>(swizzle) << 47);
  Entry& e = cache[(h ^ (h >> 29)) & (kSlots - 1)];
  if (e.valid && e.base == base && e.dim0 == dim0 && e.dim1 == dim1 && e.stride1 == stride1 && e.box0 == box0 &&
      e.box1 == box1 && e.type == static_cast<int>(type) && e.swizzle == static_cast<int>(swizzle)) {
    *map = e.map;
    return true;
  }
  auto encode = tensor_map_encoder();
  if (encode == nullptr) return false;
  cuuint64_t dims[2] = {dim0, dim1};
  cuuint64_t strides[1] = {stride1};
  cuuint32_t box[2] = {box0, box1};
  cuuint32_t elem_strides[2] = {1, 1};
  if (encode(map, type, 2, const_cast<void*>(base), dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  e = Entry{base, dim0, dim1, stride1, box0, box1, static_cast<int>(type), static_cast<int>(swizzle), true, *map};
  return true;
}

// 2-D map over the packed weight codes [n_pad, K/2] bytes: 128 x 128-byte
// boxes, 128-byte swizzle (the canonical K-major layout the MMA descriptor
// reads); columns past K/2 read as zero.
bool encode_weight_map(const void* bpacked, int64_t N, int64_t K, CUtensorMap* map) {
  const PackedLayout L = packed_layout(N, K);
  return encode_2d(CU_TENSOR_MAP_DATA_TYPE_UINT8, bpacked, static_cast<uint64_t>(K / 2),
                   static_cast<uint64_t>(L.n_pad), static_cast<uint64_t>(K / 2), kTileKBytes, kTileN,
                   CU_TENSOR_MAP_SWIZZLE_128B, map);
}

// 2-D map over the activation for one GEMM launch: bf16 [M, lda] with
// 256 x block_m boxes, no swizzle (the fused entry quantizes from shared
// memory), or codes [M, K/2] with 128-byte x block_m boxes and the 128-byte
// swizzle (landing directly in the MMA operand layout).  Rows past M and
// columns past K read as zero.

bool encode_activation_map(const void* a, int64_t M, int64_t K, int64_t lda, bool fused, int block_m,
                           CUtensorMap* map) {
  const uint32_t rows = static_cast<uint32_t>(activation_box_rows(M, block_m));
  if (fused)
    return encode_2d(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                     static_cast<uint64_t>(lda * 2), kTileK, rows, CU_TENSOR_MAP_SWIZZLE_NONE, map);
  return encode_2d(CU_TENSOR_MAP_DATA_TYPE_UINT8, a, static_cast<uint64_t>(K / 2), static_cast<uint64_t>(M),
                   static_cast<uint64_t>(K / 2), kTileKBytes, rows, CU_TENSOR_MAP_SWIZZLE_128B, map);
}

// 2-D map over the output C [M, N] bf16 for the TMA store of a whole
// [block_m x 128] tile (no swizzle; rows past M and columns past N are not
// written).  Needs N * 2 bytes per row to be a multiple of 16.
bool encode_output_map(void* c, int64_t M, int64_t N, int block_m, CUtensorMap* map) {
  if (N % 8 != 0) return false;
  return encode_2d(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c, static_cast<uint64_t>(N), static_cast<uint64_t>(M),
                   static_cast<uint64_t>(N * 2), kTileN, static_cast<uint32_t>(block_m), CU_TENSOR_MAP_SWIZZLE_NONE,
                   map);
}

// The default plan per (device, M, N, K, fused), computed once: the plan
// search queries cluster occupancy, which is too slow for every call.
void cached_default_plan(int64_t M, int64_t N, int64_t K, bool fused, const cudaDeviceProp& prop,
                         mxfp4_plan_t* plan) {
  static std::mutex mu;
  static std::map<std::tuple<int, int64_t, int64_t, int64_t, bool>, mxfp4_plan_t> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, M, N, K, fused);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *plan = it->second;
      return;
    }
  }
  default_plan(M, N, K, fused, prop, plan);
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() > 4096) cache.clear();
  cache[key] = *plan;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// The fused entry quantizes A once into a workspace and runs the GEMM on
// codes when re-reading bf16 A in every 128-row N tile costs more than the
// extra launch.  Measured on GB300: from M = 64 on, except while M <= 128 and
// those re-reads (2MK bytes per N tile) stay within ~5 MiB -- 128x4096x512
// (4 MiB) 3.55 us in one kernel against 4.1 in two, 64x3072x1536 (4.5 MiB)
// 4.4 against 5.0, while 64x7168x2048 (14 MiB) takes 6.0 in two against 11 in
// one -- and unless a tuned single-kernel plan for the exact shape measured
// faster.
constexpr int64_t kFusedRereadMax = int64_t(5) << 20;
bool two_pass_wanted(int64_t M, int64_t N, int64_t K) {
  if (M < 64 || tuned_single_kernel(M, N, K)) return false;
  return M > 128 || 2 * M * K * ((N + 127) / 128) > kFusedRereadMax;
}

size_t two_pass_workspace(int64_t M, int64_t K) {
  return align256(static_cast<size_t>(M) * static_cast<size_t>(K / 2)) +
         align256(static_cast<size_t>(M) * static_cast<size_t>(K / 32));
}


// One GEMM launch with every argument checked, its plan chosen and its tensor
// maps encoded: everything that can fail before anything is enqueued.
struct PreparedGemm {
  CUtensorMap map, amap, cmap;
  GemmArgs g;
  mxfp4_plan_t plan;
  bool fused;
};

// c_host: null, or the device address of a second [M, N] output in mapped
// host memory that the kernel writes alongside C.
mxfp4_status_t prepare_gemm(const void* a, int64_t lda, const void* as, const void* bpacked, void* C, int64_t M,
                            int64_t N, int64_t K, bool fused, const mxfp4_plan_t* user_plan, void* c_host,
                            PreparedGemm* out) {
  mxfp4_status_t st = check_mnk(M, N, K);
  if (st != MXFP4_OK) return st;
  if (a == nullptr || bpacked == nullptr || C == nullptr || (!fused && as == nullptr))
    return MXFP4_ERR_INVALID_ARG;
  if (fused && lda < K) return MXFP4_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(bpacked) || !aligned16(C) || (fused && lda % 8 != 0))
    return MXFP4_ERR_MISALIGNED;
  const DeviceInfo* dev = current_device(&st);
  if (dev == nullptr) return st;
  mxfp4_plan_t& plan = out->plan;
  if (user_plan != nullptr) {
    plan = mxfp4_plan_t{};
    plan.block_m = user_plan->block_m;
    plan.splits = user_plan->splits;
    plan.stages = user_plan->stages;
    plan.accumulators = user_plan->accumulators;
    plan.share = user_plan->share;
    if (!finish_plan(M, N, K, fused, dev->prop, &plan)) return MXFP4_ERR_INVALID_ARG;
  } else {
    cached_default_plan(M, N, K, fused, dev->prop, &plan);
    if (plan.threads == 0) return MXFP4_ERR_UNSUPPORTED_SHAPE;
  }
  out->fused = fused;
  if (!encode_weight_map(bpacked, N, K, &out->map)) return failure("cuTensorMapEncodeTiled (weights)");
  if (!encode_activation_map(a, M, K, fused ? lda : K / 2, fused, plan.block_m, &out->amap))
    return failure("cuTensorMapEncodeTiled (activation)");
  // without a K split the output tile leaves by TMA store when a map can describe C
  memset(&out->cmap, 0, sizeof(out->cmap));
  const bool c_tma = plan.splits == 1 && encode_output_map(C, M, N, plan.block_m, &out->cmap);
  GemmArgs& g = out->g;
  g = GemmArgs{};
  g.a = a;
  g.a_scales = static_cast<const uint8_t*>(as);
  const PackedLayout L = packed_layout(N, K);
  g.b_sf = static_cast<const uint8_t*>(bpacked) + L.sf_offset;
  g.c = static_cast<__nv_bfloat16*>(C);
  g.c_host = static_cast<__nv_bfloat16*>(c_host);
  g.M = static_cast<int32_t>(M);
  g.N = static_cast<int32_t>(N);
  g.K = static_cast<int32_t>(K);
  g.lda = fused ? lda : K / 2;
  g.k_tiles = static_cast<int32_t>(L.k_tiles);
  g.kt_per_split = plan.k_tiles_per_split;
  g.splits = plan.splits;
  g.stages = plan.stages;
  g.tmem_cols = static_cast<uint32_t>(plan.tmem_cols);
  g.timeout_ns = g_timeout_ns.load();
  const GemmLayout GL = gemm_layout(plan.block_m, plan.stages, plan.splits, fused, M, abf_ring_for(plan, fused, M, dev->prop));
  g.a_off = GL.a_off;
  g.abf_off = GL.abf_off;
  g.abf_stage_bytes = GL.abf_stage;
  g.abf_ring = GL.abf_ring;
  g.smem_total = GL.total;
  g.share = fused ? plan.share : 1;
  g.sfw_off = GL.sfw_off;
  g.sfa_off = GL.sfa_off;
  g.stg_off = GL.stg_off;
  g.bar_off = GL.bar_off;
  g.stg_blocks = GL.stg_blocks;
  g.a_box_rows = activation_box_rows(M, plan.block_m);
  g.accumulators = plan.accumulators;
  g.weights_early = g_programmatic.load() >= 2 ? 1 : 0;
  g.c_tma = c_tma ? 1 : 0;
  g.trigger_late = g_programmatic.load() >= 3 ? 1 : 0;
  g.err = device_error_word();
  if (g.err == nullptr) return failure("cudaGetSymbolAddress (device error word)");
  return MXFP4_OK;
}

mxfp4_status_t launch_prepared(const PreparedGemm& p, cudaStream_t stream) {
  const cudaError_t e = launch_gemm(p.map, p.amap, p.cmap, p.g, p.plan, p.fused, g_programmatic.load() != 0, stream);
  return e == cudaSuccess ? MXFP4_OK : cuda_failure("GEMM launch", e);
}

mxfp4_status_t run_gemm(const void* a, int64_t lda, const void* as, const void* bpacked, void* C, int64_t M,
                        int64_t N, int64_t K, bool fused, const mxfp4_plan_t* user_plan, cudaStream_t stream,
                        void* c_host = nullptr) {
  PreparedGemm p;
  const mxfp4_status_t st = prepare_gemm(a, lda, as, bpacked, C, M, N, K, fused, user_plan, c_host, &p);
  return st != MXFP4_OK ? st : launch_prepared(p, stream);
}

// The checks of mxfp4_quantize that need no device.
mxfp4_status_t check_quantize_args(const void* A, int64_t M, int64_t K, int64_t lda, const void* Aq,
                                   const void* As) {
  if (A == nullptr || Aq == nullptr || As == nullptr) return MXFP4_ERR_INVALID_ARG;
  if (M < 1 || K < 32 || K % 32 != 0 || lda < K) return MXFP4_ERR_INVALID_ARG;
  if (M > kMaxDim || K > kMaxDim || M * (K / 16) > (int64_t(1) << 31) * 256) return MXFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(A) || !aligned16(Aq) || lda % 8 != 0) return MXFP4_ERR_MISALIGNED;
  return MXFP4_OK;
}

// The fused layer, prepared: the GEMM launch and, on the two-pass route, the
// quantize pass in front of it.
struct PreparedQuantGemm {
  PreparedGemm gemm;
  bool two_pass = false;
  const void* A = nullptr;
  int64_t lda = 0, M = 0, K = 0;
  void *Aq = nullptr, *As = nullptr;
};

// Every check of the fused entry (and of both launches of its two-pass route),
// nothing enqueued.
mxfp4_status_t prepare_quant_gemm(const void* A, int64_t lda, const void* Bpacked, void* C, int64_t M, int64_t N,
                                  int64_t K, void* ws, size_t ws_bytes, void* c_host, PreparedQuantGemm* q) {
  mxfp4_status_t st = check_mnk(M, N, K);
  if (st != MXFP4_OK) return st;
  if (ws_bytes > 0 && ws == nullptr) return MXFP4_ERR_INVALID_ARG;
  q->two_pass = ws_bytes > 0 && two_pass_wanted(M, N, K);
  if (!q->two_pass) return prepare_gemm(A, lda, nullptr, Bpacked, C, M, N, K, true, nullptr, c_host, &q->gemm);
  if (ws_bytes < two_pass_workspace(M, K)) return MXFP4_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(ws)) return MXFP4_ERR_MISALIGNED;
  q->A = A;
  q->lda = lda;
  q->M = M;
  q->K = K;
  q->Aq = ws;
  q->As = static_cast<uint8_t*>(ws) + align256(static_cast<size_t>(M) * static_cast<size_t>(K / 2));
  st = check_quantize_args(A, M, K, lda, q->Aq, q->As);
  if (st != MXFP4_OK) return st;
  return prepare_gemm(q->Aq, K / 2, q->As, Bpacked, C, M, N, K, false, nullptr, c_host, &q->gemm);
}

mxfp4_status_t launch_quant_gemm(const PreparedQuantGemm& q, cudaStream_t s) {
  if (q.two_pass) {
    const cudaError_t e = launch_quantize(q.A, q.M, q.K, q.lda, q.Aq, q.As, g_programmatic.load() != 0, s);
    if (e != cudaSuccess) return cuda_failure("quantize launch", e);
  }
  return launch_prepared(q.gemm, s);
}

// ----------------------------------------------------------------------------- multi-layer launch
// Workspace of a multi-layer launch (every offset 256-aligned; independent of
// the device, so the size can be queried without one): per layer the
// activation codes [M, K_l/2] and scale chunks [m_tiles][k_tiles_l][1 KB],
// split-K partials for up to min(8, k_tiles_l) splits, then every counter.
struct ChainGeometry {
  int bm = 0, m_tiles = 0, layers = 0;
  struct Layer {
    int64_t N, K;
    int k_tiles, n_tiles, tiles, smax;
    size_t codes, sf, part;
    size_t done, tickets;  // counter indices
  } layer[kMaxChainLayers];
  size_t counters = 0, n_counters = 0, total = 0;
};

// 16-row tiles up to M = 32 (twice the items of 32-row ones, each quantizing
// half the rows: 32 x 4096 x 512 up/down chain 4.49 -> 4.26 us per layer),
// 64-row tiles above (32-row ones measured slower at M = 64).
int chain_block_m(int64_t M) { return M <= 32 ? 16 : 64; }

void chain_geometry(int64_t M, int64_t K, int L, const int64_t* N, ChainGeometry* g) {
  g->bm = chain_block_m(M);
  g->m_tiles = static_cast<int>(ceil_div(M, g->bm));
  g->layers = L;
  size_t off = 0, cnt = 0;
  for (int l = 0; l < L; ++l) {
    ChainGeometry::Layer& y = g->layer[l];
    y.N = N[l];
    y.K = l == 0 ? K : N[l - 1];
    y.k_tiles = static_cast<int>(ceil_div(y.K, kTileK));
    y.n_tiles = static_cast<int>(ceil_div(y.N, kTileN));
    y.tiles = y.n_tiles * g->m_tiles;
    y.smax = y.k_tiles < kMaxSplits ? y.k_tiles : kMaxSplits;
    y.codes = off;
    off += align256(static_cast<size_t>(M) * static_cast<size_t>(y.K / 2));
    y.sf = off;
    off += align256(static_cast<size_t>(g->m_tiles) * y.k_tiles * kSfTileBytes);
    y.part = off;
    if (y.smax > 1) off += align256(static_cast<size_t>(y.tiles) * y.smax * g->bm * kTileN * sizeof(float));
    y.done = cnt;
    cnt += static_cast<size_t>(g->m_tiles) * y.k_tiles;
    y.tickets = cnt;
    cnt += static_cast<size_t>(y.tiles);
  }
  g->counters = off;
  g->n_counters = cnt + 1;  // + the exit counter
  g->total = off + align256(g->n_counters * sizeof(uint32_t));
}

// The argument checks of a multi-layer launch that need no device.
mxfp4_status_t check_chain_args(const void* A, int64_t lda, int64_t M, int64_t K, int32_t L,
                                const void* const* Bpacked, const int64_t* N, void* const* C) {
  if (L < 1 || L > kMaxChainLayers || Bpacked == nullptr || N == nullptr || C == nullptr || A == nullptr)
    return MXFP4_ERR_INVALID_ARG;
  if (lda < K) return MXFP4_ERR_INVALID_ARG;
  for (int l = 0; l < L; ++l) {
    const int64_t K_l = l == 0 ? K : N[l - 1];
    mxfp4_status_t st = check_mnk(M, N[l], K_l);
    if (st != MXFP4_OK) return st;
    if (Bpacked[l] == nullptr || C[l] == nullptr) return MXFP4_ERR_INVALID_ARG;
  }
  if (!aligned16(A) || lda % 8 != 0) return MXFP4_ERR_MISALIGNED;
  for (int l = 0; l < L; ++l)
    if (!aligned16(Bpacked[l]) || !aligned16(C[l])) return MXFP4_ERR_MISALIGNED;
  return MXFP4_OK;
}

struct ChainPlan {
  int stages = 0, smem = 0, tmem_cols = 0, grid = 0;
  int splits[kMaxChainLayers];
};

// Shared memory of one CTA of the multi-layer kernel, and its tensor-memory columns.
void chain_smem(int bm, int stages, const cudaDeviceProp& prop, int* smem, int* tcols, uint32_t* offs) {
  const uint32_t st = static_cast<uint32_t>(stages);
  const uint32_t a_off = st * kTileN * kTileKBytes;
  const uint32_t sfw_off = a_off + st * static_cast<uint32_t>(bm) * kTileKBytes;
  const uint32_t sfa_off = sfw_off + st * kSfTileBytes;
  const uint32_t epi_off = sfa_off + st * 2 * kSfChunkBytes;  // the epilogue's bf16 tile [bm][128]
  const uint32_t bar_off = epi_off + static_cast<uint32_t>(bm) * kTileN * 2;
  const uint32_t total = bar_off + (3 * st + 2) * 8 + 16;
  uint32_t t = 32;
  while (t < static_cast<uint32_t>(bm + 16 * stages)) t <<= 1;
  int64_t bytes = static_cast<int64_t>(total) + 1024;
  // the same tensor-memory share rule as the single-layer kernel: CTAs that
  // fit on an SM together never ask for more than its 512 columns
  const int64_t floor_smem = (static_cast<int64_t>(prop.sharedMemPerMultiprocessor) * t + 511) / 512 -
                             static_cast<int64_t>(prop.reservedSharedMemPerBlock);
  if (bytes < floor_smem) bytes = floor_smem;
  *smem = static_cast<int>((bytes + 15) / 16 * 16);
  *tcols = static_cast<int>(t);
  if (offs != nullptr) {
    offs[0] = a_off;
    offs[1] = sfw_off;
    offs[2] = sfa_off;
    offs[3] = epi_off;
    offs[4] = bar_off;
  }
}

// Stages (the deepest ring, up to 6, that still lets two CTAs share an SM),
// then per layer the K split minimising an estimate of one item's critical
// path (~250 ns per K tile in sequence, ~700 ns for the split-K sum) among
// splits whose items all fit in one wave; the grid is the largest layer's
// item count (at most one wave).  When that grid needs at most one CTA per
// SM, the ring deepens to what one CTA per SM can hold (up to 8 stages).
bool chain_plan(const ChainGeometry& g, const cudaDeviceProp& prop, ChainPlan* pl) {
  int stages = 6, smem = 0, tcols = 0;
  for (; stages >= 2; --stages) {
    chain_smem(g.bm, stages, prop, &smem, &tcols, nullptr);
    if (2 * (static_cast<int64_t>(smem) + prop.reservedSharedMemPerBlock) <= prop.sharedMemPerMultiprocessor) break;
  }
  if (stages < 2) return false;
  static std::mutex mu;
  static std::map<std::tuple<int, int, int>, int> occ_cache;
  int dev = 0;
  cudaGetDevice(&dev);
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto key = std::make_tuple(dev, g.bm, smem);
    auto it = occ_cache.find(key);
    if (it != occ_cache.end()) {
      per_sm = it->second;
    } else {
      per_sm = chain_blocks_per_sm(g.bm, smem);
      occ_cache[key] = per_sm;
    }
  }
  if (per_sm < 1) return false;
  const int cap = per_sm * prop.multiProcessorCount;
  int grid = 1;
  for (int l = 0; l < g.layers; ++l) {
    const ChainGeometry::Layer& y = g.layer[l];
    int best = 1;
    int64_t best_cost = -1;
    for (int S = 1; S <= y.smax; ++S) {
      const int kps = static_cast<int>(ceil_div(y.k_tiles, S));
      if (ceil_div(y.k_tiles, kps) != S) continue;  // a split would be empty
      const int64_t items = static_cast<int64_t>(y.tiles) * S;
      if (S > 1 && items > cap) continue;
      const int64_t waves = ceil_div(items, cap);
      const int64_t cost = waves * kps * 250 + (S > 1 ? 700 : 0);
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        best = S;
      }
    }
    pl->splits[l] = best;
    const int64_t items = static_cast<int64_t>(y.tiles) * best;
    grid = static_cast<int>(std::max<int64_t>(grid, std::min<int64_t>(items, cap)));
  }
  // A grid of one CTA per SM at most leaves each CTA a whole SM: a deeper ring
  // (up to 8 K tiles: an item and the next layer's weights in flight).
  if (grid <= prop.multiProcessorCount) {
    for (int st = 8; st > stages; --st) {
      int sm1 = 0, tc1 = 0;
      chain_smem(g.bm, st, prop, &sm1, &tc1, nullptr);
      if (sm1 <= static_cast<int>(prop.sharedMemPerBlockOptin) && tc1 <= 512 && chain_blocks_per_sm(g.bm, sm1) >= 1) {
        stages = st;
        smem = sm1;
        tcols = tc1;
        break;
      }
    }
  }
  pl->stages = stages;
  pl->smem = smem;
  pl->tmem_cols = tcols;
  pl->grid = grid;
  return true;
}

}  // namespace

void set_last_error(const char* what) { snprintf(g_last_error, sizeof(g_last_error), "%s", what); }

mxfp4_status_t check_mnk(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || N < 1 || K < 32 || K % 32 != 0) return MXFP4_ERR_INVALID_ARG;
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return MXFP4_ERR_UNSUPPORTED_SHAPE;
  // 32-bit indices and grid limits inside the kernels
  if (M * N > (int64_t(1) << 31) || K / 2 * ceil_div(N, kTileN) * kTileN > (int64_t(1) << 40) ||
      M > 65535LL * 256)
    return MXFP4_ERR_UNSUPPORTED_SHAPE;
  return MXFP4_OK;
}

mxfp4_status_t check_device() {
  mxfp4_status_t st;
  current_device(&st);
  return st;
}

mxfp4_status_t two_pass(const void* A, int64_t lda, const void* Bpacked, void* C, int64_t M, int64_t N, int64_t K,
                        void* Aq, void* As, cudaStream_t s, void* c_host) {
  // Every check of both launches first (the GEMM's plan and tensor maps
  // included), so that an error status means nothing was launched.
  mxfp4_status_t st = check_mnk(M, N, K);
  if (st != MXFP4_OK) return st;
  PreparedQuantGemm q;
  q.two_pass = true;
  q.A = A;
  q.lda = lda;
  q.M = M;
  q.K = K;
  q.Aq = Aq;
  q.As = As;
  st = check_quantize_args(A, M, K, lda, Aq, As);
  if (st != MXFP4_OK) return st;
  st = prepare_gemm(Aq, K / 2, As, Bpacked, C, M, N, K, false, nullptr, c_host, &q.gemm);
  if (st != MXFP4_OK) return st;
  return launch_quant_gemm(q, s);
}

}  // namespace mxfp4

using namespace mxfp4;

extern "C" {

mxfp4_status_t mxfp4_quantize(const void* A, int64_t M, int64_t K, int64_t lda, void* Aq, void* As,
                              mxfp4_stream_t stream) {
  mxfp4_status_t st = check_quantize_args(A, M, K, lda, Aq, As);
  if (st != MXFP4_OK) return st;
  if (current_device(&st) == nullptr) return st;
  const cudaError_t e =
      launch_quantize(A, M, K, lda, Aq, As, g_programmatic.load() != 0, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXFP4_OK : cuda_failure("quantize launch", e);
}

size_t mxfp4_packed_weight_bytes(int64_t N, int64_t K) {
  if (N < 1 || K < 32 || K % 32 != 0 || N > kMaxDim || K > kMaxDim) return 0;
  return packed_layout(N, K).total;
}

mxfp4_status_t mxfp4_pack_weights(const void* Bq, const void* Bs, int64_t N, int64_t K, void* Bpacked,
                                  mxfp4_stream_t stream) {
  if (Bq == nullptr || Bs == nullptr || Bpacked == nullptr) return MXFP4_ERR_INVALID_ARG;
  if (N < 1 || K < 32 || K % 32 != 0) return MXFP4_ERR_INVALID_ARG;
  if (N > kMaxDim || K > kMaxDim) return MXFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(Bq) || !aligned16(Bpacked)) return MXFP4_ERR_MISALIGNED;
  mxfp4_status_t st;
  if (current_device(&st) == nullptr) return st;
  const cudaError_t e = launch_pack_weights(Bq, Bs, N, K, Bpacked, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXFP4_OK : cuda_failure("weight packing launch", e);
}

mxfp4_status_t mxfp4_pack_weights_shuffled(const void* B_shuffle, const void* B_scale_sh, int64_t N, int64_t K,
                                           void* Bpacked, mxfp4_stream_t stream) {
  if (B_shuffle == nullptr || B_scale_sh == nullptr || Bpacked == nullptr) return MXFP4_ERR_INVALID_ARG;
  if (N < 1 || K < 64 || N % 16 != 0 || K % 64 != 0) return MXFP4_ERR_INVALID_ARG;
  if (N > kMaxDim || K > kMaxDim) return MXFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(Bpacked)) return MXFP4_ERR_MISALIGNED;
  mxfp4_status_t st;
  if (current_device(&st) == nullptr) return st;
  const cudaError_t e =
      launch_pack_from_shuffled(B_shuffle, B_scale_sh, N, K, Bpacked, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXFP4_OK : cuda_failure("shuffled weight packing launch", e);
}

mxfp4_status_t mxfp4_unpack_weights(const void* Bpacked, int64_t N, int64_t K, void* Bq, void* Bs,
                                    mxfp4_stream_t stream) {
  if (Bq == nullptr || Bs == nullptr || Bpacked == nullptr) return MXFP4_ERR_INVALID_ARG;
  if (N < 1 || K < 32 || K % 32 != 0) return MXFP4_ERR_INVALID_ARG;
  if (N > kMaxDim || K > kMaxDim) return MXFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(Bq) || !aligned16(Bpacked)) return MXFP4_ERR_MISALIGNED;
  mxfp4_status_t st;
  if (current_device(&st) == nullptr) return st;
  const cudaError_t e = launch_unpack_weights(Bpacked, N, K, Bq, Bs, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXFP4_OK : cuda_failure("weight unpacking launch", e);
}

size_t mxfp4_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (check_mnk(M, N, K) != MXFP4_OK) return 0;
  return two_pass_wanted(M, N, K) ? two_pass_workspace(M, K) : 0;
}

mxfp4_status_t mxfp4_gemm(const void* Aq, const void* As, const void* Bpacked, void* C, int64_t M,
                          int64_t N, int64_t K, void* ws, size_t ws_bytes, mxfp4_stream_t stream) {
  (void)ws;
  (void)ws_bytes;  // the pre-quantized GEMM needs no scratch
  return run_gemm(Aq, K / 2, As, Bpacked, C, M, N, K, false, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

mxfp4_status_t mxfp4_quant_gemm(const void* A, int64_t lda, const void* Bpacked, void* C, int64_t M,
                                int64_t N, int64_t K, void* ws, size_t ws_bytes, mxfp4_stream_t stream) {
  PreparedQuantGemm q;
  const mxfp4_status_t st = prepare_quant_gemm(A, lda, Bpacked, C, M, N, K, ws, ws_bytes, nullptr, &q);
  return st != MXFP4_OK ? st : launch_quant_gemm(q, reinterpret_cast<cudaStream_t>(stream));
}

mxfp4_status_t mxfp4_quant_gemm_host(const void* A_host, int64_t lda_host, void* A_dev, int64_t lda_dev,
                                     const void* Bpacked, void* C_dev, void* C_host, int64_t M, int64_t N,
                                     int64_t K, void* ws, size_t ws_bytes, mxfp4_stream_t stream) {
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mxfp4_status_t st = check_mnk(M, N, K);
  if (st != MXFP4_OK) return st;
  if (A_host == nullptr || C_host == nullptr || A_dev == nullptr) return MXFP4_ERR_INVALID_ARG;
  if (lda_host < K) return MXFP4_ERR_INVALID_ARG;
  // A mapped C_host is written by the GEMM kernel itself, beside C_dev (no
  // download pass); any other by the copy engines afterwards.
  void* c_dst = const_cast<void*>(device_view(C_host));
  const bool c_direct = c_dst != nullptr && aligned16(c_dst);
  // every check of the layer (both routes, plan and tensor maps included)
  // before the upload, so that an error launches nothing
  PreparedQuantGemm q;
  st = prepare_quant_gemm(A_dev, lda_dev, Bpacked, C_dev, M, N, K, ws, ws_bytes, c_direct ? c_dst : nullptr, &q);
  if (st != MXFP4_OK) return st;
  const DeviceInfo* dev = current_device(&st);
  if (dev == nullptr) return st;
  const bool programmatic = g_programmatic.load() != 0;
  const int sms = dev->prop.multiProcessorCount;
  // Pinned, mapped host buffers are moved by SM threads over the host link;
  // anything else (pageable memory, unaligned rows) by the copy engines.
  const void* a_src = device_view(A_host);
  cudaError_t e;
  if (a_src != nullptr && aligned16(a_src) && lda_host % 8 == 0) {
    e = launch_copy_rows(a_src, lda_host * 2, A_dev, lda_dev * 2, K * 2, M, true, programmatic, sms, s);
  } else {
    e = cudaMemcpy2DAsync(A_dev, static_cast<size_t>(lda_dev) * 2, A_host, static_cast<size_t>(lda_host) * 2,
                          static_cast<size_t>(K) * 2, static_cast<size_t>(M), cudaMemcpyHostToDevice, s);
  }
  if (e != cudaSuccess) return cuda_failure("activation upload", e);
  st = launch_quant_gemm(q, s);
  if (st != MXFP4_OK || c_direct) return st;
  e = cudaMemcpyAsync(C_host, C_dev, static_cast<size_t>(M * N * 2), cudaMemcpyDeviceToHost, s);
  return e == cudaSuccess ? MXFP4_OK : cuda_failure("result download", e);
}

mxfp4_status_t mxfp4_gemm_plan(int64_t M, int64_t N, int64_t K, int fused, mxfp4_plan_t* plan) {
  if (plan == nullptr) return MXFP4_ERR_INVALID_ARG;
  mxfp4_status_t st = check_mnk(M, N, K);
  if (st != MXFP4_OK) return st;
  const DeviceInfo* dev = current_device(&st);
  if (dev == nullptr) return st;
  const bool two_pass = fused != 0 && two_pass_wanted(M, N, K);
  cached_default_plan(M, N, K, fused != 0 && !two_pass, dev->prop, plan);
  plan->two_pass = two_pass ? 1 : 0;
  return plan->threads == 0 ? MXFP4_ERR_UNSUPPORTED_SHAPE : MXFP4_OK;
}

mxfp4_status_t mxfp4_gemm_with_plan(const void* A_or_Aq, int64_t lda, const void* As, const void* Bpacked,
                                    void* C, int64_t M, int64_t N, int64_t K, int fused,
                                    const mxfp4_plan_t* plan, mxfp4_stream_t stream) {
  if (plan == nullptr) return MXFP4_ERR_INVALID_ARG;
  return run_gemm(A_or_Aq, fused ? lda : K / 2, As, Bpacked, C, M, N, K, fused != 0, plan,
                  reinterpret_cast<cudaStream_t>(stream));
}

size_t mxfp4_chain_workspace_bytes(int64_t M, int64_t K, int32_t num_layers, const int64_t* N) {
  if (num_layers < 1 || num_layers > kMaxChainLayers || N == nullptr) return 0;
  for (int l = 0; l < num_layers; ++l) {
    const int64_t K_l = l == 0 ? K : N[l - 1];
    if (check_mnk(M, N[l], K_l) != MXFP4_OK) return 0;
  }
  ChainGeometry g;
  chain_geometry(M, K, num_layers, N, &g);
  return g.total;
}

mxfp4_status_t mxfp4_quant_gemm_chain(const void* A, int64_t lda, int64_t M, int64_t K, int32_t num_layers,
                                      const void* const* Bpacked, const int64_t* N, void* const* C, void* ws,
                                      size_t ws_bytes, mxfp4_stream_t stream) {
  mxfp4_status_t st = check_chain_args(A, lda, M, K, num_layers, Bpacked, N, C);
  if (st != MXFP4_OK) return st;
  ChainGeometry g;
  chain_geometry(M, K, num_layers, N, &g);
  if (ws == nullptr) return MXFP4_ERR_INVALID_ARG;
  if (ws_bytes < g.total) return MXFP4_ERR_WORKSPACE_TOO_SMALL;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MXFP4_ERR_MISALIGNED;
  const DeviceInfo* dev = current_device(&st);
  if (dev == nullptr) return st;
  ChainPlan pl;
  if (!chain_plan(g, dev->prop, &pl)) return MXFP4_ERR_UNSUPPORTED_SHAPE;
  uint8_t* base = static_cast<uint8_t*>(ws);
  uint32_t* counters = reinterpret_cast<uint32_t*>(base + g.counters);
  ChainArgs a;
  memset(&a, 0, sizeof(a));
  for (int l = 0; l < num_layers; ++l) {
    const ChainGeometry::Layer& y = g.layer[l];
    ChainLayerArgs& L = a.layer[l];
    if (!encode_weight_map(Bpacked[l], y.N, y.K, &a.wmap[l])) return failure("cuTensorMapEncodeTiled (weights)");
    if (!encode_activation_map(base + y.codes, M, y.K, y.K / 2, false, g.bm, &a.amap[l]))
      return failure("cuTensorMapEncodeTiled (activation codes)");
    L.b_sf = static_cast<const uint8_t*>(Bpacked[l]) + packed_layout(y.N, y.K).sf_offset;
    L.c = static_cast<__nv_bfloat16*>(C[l]);
    L.in_sf = base + y.sf;
    L.in_done = counters + y.done;
    L.in_n_tiles = l == 0 ? 0 : g.layer[l - 1].n_tiles;
    L.in_splits = l == 0 ? 1 : pl.splits[l - 1];
    if (l + 1 < num_layers) {
      const ChainGeometry::Layer& nx = g.layer[l + 1];
      L.out_codes = base + nx.codes;
      L.out_sf = base + nx.sf;
      L.out_done = counters + nx.done;
      L.k_tiles_next = nx.k_tiles;
    }
    L.partials = reinterpret_cast<float*>(base + y.part);
    L.tickets = counters + y.tickets;
    L.N = static_cast<int32_t>(y.N);
    L.K = static_cast<int32_t>(y.K);
    L.k_tiles = y.k_tiles;
    L.splits = pl.splits[l];
    L.kt_per_split = static_cast<int32_t>(ceil_div(y.k_tiles, pl.splits[l]));
    L.n_tiles = y.n_tiles;
    L.items = y.tiles * pl.splits[l];
  }
  a.a = static_cast<const uint16_t*>(A);
  a.lda = lda;
  a.a_codes = base + g.layer[0].codes;
  a.a_sf = base + g.layer[0].sf;
  a.a_done = counters + g.layer[0].done;
  a.counters = counters;
  a.n_counters = static_cast<int32_t>(g.n_counters);
  a.exit_count = counters + (g.n_counters - 1);
  a.err = device_error_word();
  if (a.err == nullptr) return failure("cudaGetSymbolAddress (device error word)");
  a.timeout_ns = g_timeout_ns.load();
  a.layers = num_layers;
  a.M = static_cast<int32_t>(M);
  a.K0 = static_cast<int32_t>(K);
  a.k_tiles0 = g.layer[0].k_tiles;
  a.m_tiles = g.m_tiles;
  a.stages = pl.stages;
  a.a_box_rows = activation_box_rows(M, g.bm);
  a.tmem_cols = static_cast<uint32_t>(pl.tmem_cols);
  uint32_t offs[5];
  int smem = 0, tcols = 0;
  chain_smem(g.bm, pl.stages, dev->prop, &smem, &tcols, offs);
  a.a_off = offs[0];
  a.sfw_off = offs[1];
  a.sfa_off = offs[2];
  a.epi_off = offs[3];
  a.bar_off = offs[4];
  a.weights_early = g_programmatic.load() >= 2 ? 1 : 0;
  const cudaError_t e = launch_chain(a, g.bm, pl.grid, pl.smem, g_programmatic.load() != 0,
                                     reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXFP4_OK : cuda_failure("multi-layer launch", e);
}

mxfp4_status_t mxfp4_chain_plan(int64_t M, int64_t K, int32_t num_layers, const int64_t* N, int32_t* splits,
                                int32_t* grid, int32_t* block_m) {
  if (num_layers < 1 || num_layers > kMaxChainLayers || N == nullptr) return MXFP4_ERR_INVALID_ARG;
  for (int l = 0; l < num_layers; ++l) {
    const int64_t K_l = l == 0 ? K : N[l - 1];
    mxfp4_status_t st = check_mnk(M, N[l], K_l);
    if (st != MXFP4_OK) return st;
  }
  mxfp4_status_t st;
  const DeviceInfo* dev = current_device(&st);
  if (dev == nullptr) return st;
  ChainGeometry g;
  chain_geometry(M, K, num_layers, N, &g);
  ChainPlan pl;
  if (!chain_plan(g, dev->prop, &pl)) return MXFP4_ERR_UNSUPPORTED_SHAPE;
  for (int l = 0; l < num_layers && splits != nullptr; ++l) splits[l] = pl.splits[l];
  if (grid != nullptr) *grid = pl.grid;
  if (block_m != nullptr) *block_m = g.bm;
  return MXFP4_OK;
}

const char* mxfp4_status_string(mxfp4_status_t status) {
  switch (status) {
    case MXFP4_OK: return "ok";
    case MXFP4_ERR_INVALID_ARG: return "invalid argument";
    case MXFP4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MXFP4_ERR_MISALIGNED: return "pointer or leading dimension not 16-byte aligned";
    case MXFP4_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MXFP4_ERR_CUDA: return "CUDA error";
    case MXFP4_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out";
    case MXFP4_ERR_UNSUPPORTED_DEVICE: return "current device is not sm_103 (GB300)";
  }
  return "unknown status";
}

mxfp4_status_t mxfp4_device_error(mxfp4_stream_t stream, int reset, uint32_t* code) {
  if (code == nullptr) return MXFP4_ERR_INVALID_ARG;
  mxfp4_status_t st;
  if (current_device(&st) == nullptr) return st;
  const cudaError_t e = read_device_error(reinterpret_cast<cudaStream_t>(stream), code, reset != 0);
  if (e != cudaSuccess) return cuda_failure("reading the device error word", e);
  return *code != 0 ? MXFP4_ERR_DEVICE_TIMEOUT : MXFP4_OK;
}

const char* mxfp4_last_error_string(void) { return g_last_error; }

mxfp4_status_t mxfp4_set_wait_timeout_ns(uint64_t ns) {
  g_timeout_ns.store(ns == 0 ? 1000000000ull : ns);
  return MXFP4_OK;
}

mxfp4_status_t mxfp4_set_programmatic_launch(int mode) {
  if (mode < 0 || mode > 3) return MXFP4_ERR_INVALID_ARG;
  g_programmatic.store(mode);
  return MXFP4_OK;
}

mxfp4_status_t mxfp4_diag_wait_timeout(mxfp4_stream_t stream) {
  mxfp4_status_t st;
  if (current_device(&st) == nullptr) return st;
  const cudaError_t e = launch_diag_wait(g_timeout_ns.load(), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXFP4_OK : cuda_failure("diagnostic launch", e);
}

}  // extern "C"
