// Standalone kernels: activation quantization, the one-time weight relayout
// and its inverse, the bounded-wait diagnostic, and the device error word.
#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace mxfp4 {

// The device error word; kernels receive its address as an argument.
static __device__ uint32_t g_device_error = 0;

uint32_t* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  static uint32_t* cache[64] = {};
  if (cache[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<uint32_t*>(p);
  }
  return cache[dev];
}

// ----------------------------------------------------------------------------- quantize
// One thread per 16 consecutive elements of a row (two 16-byte loads in
// flight); 2 lanes per 32-element block, combining their maxima with one
// shuffle; a warp covers 512 consecutive elements (1 KB of A).  Rows are K/16
// units long and K % 32 == 0, so a block never straddles two rows and both
// lanes of a block are always in or out of range together.  (On GB300 this
// beat 4 lanes of 8 elements by ~0.25 us per call at M = 64 and 256: half the
// threads, the same load latency.)
__global__ void __launch_bounds__(256) quantize_kernel(const uint16_t* __restrict__ A, int64_t M,
                                                       int64_t K, int64_t lda,
                                                       uint8_t* __restrict__ Aq,
                                                       uint8_t* __restrict__ As, uint32_t* err) {
  const int64_t units_per_row = K / 16;
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const bool valid = unit < M * units_per_row;
  const int64_t row = valid ? unit / units_per_row : 0;
  const int64_t j = valid ? unit - row * units_per_row : 0;
  const uint16_t* src = A + row * lda + j * 16;
  // Under programmatic launch the next kernel may start its prologue now; this
  // one touches A and its outputs only once the previous grid has completed
  // (the outputs may still be read by it), after an L2 prefetch of its line.
  grid_launch_dependents();
  if (valid && (j & 3) == 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(src));
  grid_dependency_wait();
  uint4 v = make_uint4(0, 0, 0, 0), w = make_uint4(0, 0, 0, 0);
  if (valid && MXFP4_IN_BOUNDS(row * lda + j * 16 + 16 <= M * lda, err)) {
    v = ld_after_wait_v4(src);  // A may be the previous grid's output
    w = ld_after_wait_v4(src + 8);
  }
  // every lane takes part in the shuffle
  uint32_t amax = absmax16_bf16(v, w);
  amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  const uint32_t byte = scale_byte_from_amax(amax);
  const uint16_t sbf = scale_bf16_from_byte(byte);
  const uint32_t c0 = e2m1_pack8(v, sbf), c1 = e2m1_pack8(w, sbf);
  if (valid && MXFP4_IN_BOUNDS(row * (K / 2) + j * 8 + 8 <= M * (K / 2), err)) {
    *reinterpret_cast<uint2*>(Aq + row * (K / 2) + j * 8) = make_uint2(c0, c1);
    if ((j & 1) == 0) As[row * (K / 32) + j / 2] = static_cast<uint8_t>(byte);
  }
}

cudaError_t launch_quantize(const void* A, int64_t M, int64_t K, int64_t lda, void* Aq, void* As,
                            bool programmatic, cudaStream_t s) {
  const int64_t units = M * (K / 16);
  const int threads = 256;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(units, threads)), 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = programmatic ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quantize_kernel, static_cast<const uint16_t*>(A), M, K, lda,
                            static_cast<uint8_t*>(Aq), static_cast<uint8_t*>(As), device_error_word());
}

// ----------------------------------------------------------------------------- weight relayout
// Position of scale (n, j) -- row n, 32-element block j -- in the packed scale
// region: tile (n / 128, j / 8), chunk (j % 8) / 4, byte (r % 32) * 16 +
// (r / 32) * 4 + j % 4 with r = n % 128.  This is the 128-row x 4-scale chunk
// that one tcgen05.cp 32x128b.warpx4 moves into tensor memory.
__device__ __forceinline__ size_t packed_sf_index(int64_t n, int64_t j, int64_t k_tiles) {
  const int64_t tile = (n / kTileN) * k_tiles + j / 8;
  const int64_t r = n % kTileN;
  return static_cast<size_t>(tile) * kSfTileBytes + ((j % 8) / 4) * kSfChunkBytes + (r % 32) * 16 +
         (r / 32) * 4 + (j % 4);
}

__global__ void pack_codes_kernel(const uint4* __restrict__ bq, int64_t N, int64_t n_pad,
                                  int64_t row_vecs, uint4* __restrict__ out) {
  const int64_t total = n_pad * row_vecs;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t n = i / row_vecs;
    out[i] = (n < N) ? bq[i] : make_uint4(0, 0, 0, 0);
  }
}

__global__ void pack_scales_kernel(const uint8_t* __restrict__ bs, int64_t N, int64_t n_pad,
                                   int64_t nblk, int64_t k_tiles, uint8_t* __restrict__ sf) {
  const int64_t per_row = k_tiles * 8;
  const int64_t total = n_pad * per_row;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t n = i / per_row, j = i % per_row;
    sf[packed_sf_index(n, j, k_tiles)] = (n < N && j < nblk) ? bs[n * nblk + j] : 0;
  }
}

__global__ void unpack_kernel(const uint8_t* __restrict__ bp, int64_t N, int64_t K, size_t sf_offset,
                              int64_t k_tiles, uint8_t* __restrict__ bq, uint8_t* __restrict__ bs) {
  const int64_t kh = K / 2, nblk = K / 32;
  const int64_t total = N * kh;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    bq[i] = bp[i];
    const int64_t n = i / kh, b = i % kh;
    if (b % 16 == 0) bs[n * nblk + b / 16] = bp[sf_offset + packed_sf_index(n, b / 16, k_tiles)];
  }
}

// ----------------------------------------------------------------------------- ingest of the pages' layouts
// Weight codes in the pages' preshuffled layout (submission 748756,
// `materialize_linear_weight_layout`): 16-row x 16-byte subtiles, byte (n, kb)
// of the natural [N, K/2] array at ((n/16 * Kh/32 + kb/32) * 2 + (kb%32)/16)
// * 256 + (n%16) * 16 + kb%16, Kh = K/2.  Scales in the e8m0 shuffle (the
// store of submission 755056's standalone quantizer, inverted by
// `materialize_linear_scale_layout`): scale (n, g) at (n/32) * 32 * Gp +
// (g/8) * 256 + (g%4) * 64 + (n%16) * 4 + ((g%8)/4) * 2 + (n%32)/16, Gp = K/32
// rounded up to 8.
__device__ __forceinline__ int64_t shuffled_code_index(int64_t n, int64_t kb, int64_t kh) {
  return ((n / 16 * (kh / 32) + kb / 32) * 2 + (kb % 32) / 16) * 256 + (n % 16) * 16 + kb % 16;
}

__device__ __forceinline__ int64_t shuffled_scale_index(int64_t n, int64_t g, int64_t gp) {
  return (n / 32) * 32 * gp + (g / 8) * 256 + (g % 4) * 64 + (n % 16) * 4 + ((g % 8) / 4) * 2 + (n % 32) / 16;
}

__global__ void pack_from_shuffled_kernel(const uint8_t* __restrict__ bsh, const uint8_t* __restrict__ ssh,
                                          int64_t N, int64_t K, int64_t n_pad, int64_t k_tiles,
                                          uint8_t* __restrict__ out, size_t sf_offset) {
  const int64_t kh = K / 2, nblk = K / 32, gp = (nblk + 7) / 8 * 8;
  const int64_t codes = n_pad * kh, scales = n_pad * k_tiles * 8;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < codes + scales;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (i < codes) {
      const int64_t n = i / kh, kb = i % kh;
      out[i] = n < N ? bsh[shuffled_code_index(n, kb, kh)] : 0;
    } else {
      const int64_t j = i - codes, n = j / (k_tiles * 8), g = j % (k_tiles * 8);
      out[sf_offset + packed_sf_index(n, g, k_tiles)] = (n < N && g < nblk) ? ssh[shuffled_scale_index(n, g, gp)] : 0;
    }
  }
}

static unsigned grid_for(int64_t work, int threads) {
  int64_t b = ceil_div(work, threads);
  if (b > 65536) b = 65536;
  if (b < 1) b = 1;
  return static_cast<unsigned>(b);
}

cudaError_t launch_pack_weights(const void* Bq, const void* Bs, int64_t N, int64_t K, void* Bp,
                                cudaStream_t s) {
  const PackedLayout L = packed_layout(N, K);
  uint8_t* out = static_cast<uint8_t*>(Bp);
  const int64_t row_vecs = K / 32;  // 16-byte vectors per row of codes
  pack_codes_kernel<<<grid_for(L.n_pad * row_vecs, 256), 256, 0, s>>>(
      static_cast<const uint4*>(Bq), N, L.n_pad, row_vecs, reinterpret_cast<uint4*>(out));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (L.sf_offset > L.data_bytes) {
    e = cudaMemsetAsync(out + L.data_bytes, 0, L.sf_offset - L.data_bytes, s);
    if (e != cudaSuccess) return e;
  }
  pack_scales_kernel<<<grid_for(L.n_pad * L.k_tiles * 8, 256), 256, 0, s>>>(
      static_cast<const uint8_t*>(Bs), N, L.n_pad, K / 32, L.k_tiles, out + L.sf_offset);
  return cudaGetLastError();
}

cudaError_t launch_pack_from_shuffled(const void* Bsh, const void* Ssh, int64_t N, int64_t K, void* Bp,
                                      cudaStream_t s) {
  const PackedLayout L = packed_layout(N, K);
  uint8_t* out = static_cast<uint8_t*>(Bp);
  if (L.sf_offset > L.data_bytes) {
    const cudaError_t e = cudaMemsetAsync(out + L.data_bytes, 0, L.sf_offset - L.data_bytes, s);
    if (e != cudaSuccess) return e;
  }
  const int64_t work = L.n_pad * (K / 2) + L.n_pad * L.k_tiles * 8;
  pack_from_shuffled_kernel<<<grid_for(work, 256), 256, 0, s>>>(static_cast<const uint8_t*>(Bsh),
                                                               static_cast<const uint8_t*>(Ssh), N, K, L.n_pad,
                                                               L.k_tiles, out, L.sf_offset);
  return cudaGetLastError();
}

cudaError_t launch_unpack_weights(const void* Bp, int64_t N, int64_t K, void* Bq, void* Bs,
                                  cudaStream_t s) {
  const PackedLayout L = packed_layout(N, K);
  unpack_kernel<<<grid_for(N * (K / 2), 256), 256, 0, s>>>(
      static_cast<const uint8_t*>(Bp), N, K, L.sf_offset, L.k_tiles, static_cast<uint8_t*>(Bq),
      static_cast<uint8_t*>(Bs));
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------- diagnostics
// Waits on an mbarrier that expects two arrivals and gets one, so its phase
// never completes; the bounded wait gives up after timeout_ns and reports.
__global__ void diag_wait_kernel(uint64_t timeout_ns, uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 2);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive(b);
    if (!mbar_wait(b, 0, timeout_ns)) report_error(err, kErrDiag);
  }
}

cudaError_t launch_diag_wait(uint64_t timeout_ns, cudaStream_t s) {
  uint32_t* err = device_error_word();
  if (err == nullptr) return cudaErrorInvalidSymbol;
  diag_wait_kernel<<<1, 32, 0, s>>>(timeout_ns, err);
  return cudaGetLastError();
}

cudaError_t read_device_error(cudaStream_t s, uint32_t* code, bool reset) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  uint32_t v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
  if (e != cudaSuccess) return e;
  if (reset && v != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
  }
  *code = v;
  return cudaSuccess;
}

}  // namespace mxfp4
