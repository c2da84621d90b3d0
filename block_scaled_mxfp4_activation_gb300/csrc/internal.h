// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "mxfp4.h"

namespace mxfp4 {

// Geometry shared by the packed-weight layout and the GEMM kernel.
constexpr int kTileN = 128;                      // weight rows per CTA (the MMA's M)
constexpr int kTileK = 256;                      // K elements per pipeline stage
constexpr int kTileKBytes = kTileK / 2;          // 128 bytes of codes per row and stage
constexpr int kSfChunkBytes = 512;               // 128 rows x 4 scales
constexpr int kSfTileBytes = 2 * kSfChunkBytes;  // scales of one 128 x 256 weight tile
constexpr int kMaxSplits = 8;                    // portable cluster size

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Largest M, N or K any entry accepts.
constexpr int64_t kMaxDim = int64_t(1) << 30;

struct PackedLayout {
  int64_t n_pad;     // rows rounded up to kTileN
  int64_t k_tiles;   // ceil(K / kTileK)
  size_t data_bytes; // n_pad * K / 2
  size_t sf_offset;  // data_bytes rounded up to 1024
  size_t sf_bytes;   // (n_pad / kTileN) * k_tiles * kSfTileBytes
  size_t total;
};

inline PackedLayout packed_layout(int64_t N, int64_t K) {
  PackedLayout L;
  L.n_pad = ceil_div(N, kTileN) * kTileN;
  L.k_tiles = ceil_div(K, kTileK);
  L.data_bytes = static_cast<size_t>(L.n_pad) * static_cast<size_t>(K / 2);
  L.sf_offset = (L.data_bytes + 1023) / 1024 * 1024;
  L.sf_bytes = static_cast<size_t>(L.n_pad / kTileN) * static_cast<size_t>(L.k_tiles) * kSfTileBytes;
  L.total = L.sf_offset + L.sf_bytes;
  return L;
}

struct GemmArgs {
  const void* a;            // fused: bf16 A [M, lda]; else codes Aq [M, K/2]
  const uint8_t* a_scales;  // unfused: As [M, K/32]
  const uint8_t* b_sf;      // packed weight scales
  __nv_bfloat16* c;         // [M, N]
  __nv_bfloat16* c_host;    // or null: a second copy of C, [M, N] in mapped host memory (device address)
  int32_t M, N, K;
  int64_t lda;              // fused: elements per row of A
  int32_t k_tiles;          // ceil(K / kTileK)
  int32_t kt_per_split;
  int32_t splits;
  int32_t stages;
  uint32_t tmem_cols;
  uint64_t timeout_ns;
  uint32_t* err;            // device error word
  int32_t weights_early;    // issue the weight loads before waiting on the previous grid
  // shared-memory layout (byte offsets from the 1024-aligned base), see smem_layout()
  uint32_t a_off, abf_off, sfw_off, sfa_off, stg_off, bar_off;
  int32_t stg_blocks;       // 32 x 16 partial blocks each CTA may receive from one split
  int32_t a_box_rows;       // rows of one activation TMA box: min(block_m, roundup(M, 8))
  uint32_t abf_stage_bytes; // fused: bf16 staging per stage, a_box_rows x 512 bytes
  int32_t accumulators;     // independent fp32 accumulator tiles in tensor memory (1, 2, 4)
  int32_t c_tma;            // no K split: C leaves through a bf16 tile in shared memory and one TMA store
  int32_t trigger_late;     // let the next grid launch only once this grid has passed its own wait
  int32_t abf_ring;         // fused: bf16 staging buffers (a ring of its own, at most kAbfRing)
  int32_t share;            // CTAs along N sharing the quantization of their rows (1: none)
  uint32_t smem_total;      // bytes of the shared-memory layout (bounds of the checked build)
};

// bf16 activation buffers of the fused kernel: tile i is staged in buffer
// i % ring and the buffer is refilled once that tile is quantized, so the
// stage count (weight tiles in flight) does not pay for bf16 staging; the
// ring holds all of a split's K tiles up to this many.
constexpr int kAbfRing = 4;

// Shared-memory layout of one GEMM CTA (byte offsets from a 1024-aligned base):
// weight code tiles, activation code tiles, bf16 activation staging (fused,
// activation_box_rows x 512 bytes per buffer, min(K tiles per split, kAbfRing) buffers),
// weight scales, activation scales (one of each per stage), the split-K
// staging slots ([splits][stg_blocks] blocks of 2 KB), then the mbarriers.
// Without a K split the bf16 output tile [block_m][128] is staged at offset 0
// once the MMAs are done (the operand buffers are free by then); the layout
// keeps at least block_m x 256 bytes before the scales for it.
// Rows of one activation TMA box (and of the bf16 staging): the tile's rows
// that can hold data, rounded up to 8.
inline int activation_box_rows(int64_t M, int block_m) {
  const int64_t r = (M + 7) / 8 * 8;
  return static_cast<int>(r < block_m ? r : block_m);
}

struct GemmLayout {
  uint32_t a_off, abf_off, sfw_off, sfa_off, stg_off, bar_off, total;
  uint32_t abf_stage;  // bf16 staging bytes per buffer (fused)
  int32_t abf_ring;    // bf16 staging buffers (fused)
  int32_t stg_blocks;
};
GemmLayout gemm_layout(int block_m, int stages, int splits, bool fused, int64_t M, int abf_ring);
// True when the tuned plans hold a single fused-kernel plan for this exact
// shape (the fused entry then takes no two-pass route, whatever M).
bool tuned_single_kernel(int64_t M, int64_t N, int64_t K);
// The fused kernel's bf16 buffer count for a finished plan (0 unfused).
int abf_ring_for(const mxfp4_plan_t& p, bool fused, int64_t M, const cudaDeviceProp& prop);

// Launchers (return a CUDA error code; arguments are validated by the caller).
cudaError_t launch_quantize(const void* A, int64_t M, int64_t K, int64_t lda, void* Aq, void* As,
                            bool programmatic, cudaStream_t s);
cudaError_t launch_pack_weights(const void* Bq, const void* Bs, int64_t N, int64_t K, void* Bp,
                                cudaStream_t s);
cudaError_t launch_pack_from_shuffled(const void* Bsh, const void* Ssh, int64_t N, int64_t K, void* Bp,
                                      cudaStream_t s);
// Row copy by SM threads between device-addressable buffers (row_bytes, pitches
// and addresses multiples of 16); see host_copy.cu.
cudaError_t launch_copy_rows(const void* src, int64_t src_pitch, void* dst, int64_t dst_pitch, int64_t row_bytes,
                             int64_t rows, bool src_early, bool programmatic, int sm_count, cudaStream_t s);
cudaError_t launch_unpack_weights(const void* Bp, int64_t N, int64_t K, void* Bq, void* Bs,
                                  cudaStream_t s);
cudaError_t launch_diag_wait(uint64_t timeout_ns, cudaStream_t s);

// Fills the derived fields of a plan (block_m, splits, stages given).
// Returns false if the plan cannot run.
bool finish_plan(int64_t M, int64_t N, int64_t K, bool fused, const cudaDeviceProp& prop,
                 mxfp4_plan_t* plan);
void default_plan(int64_t M, int64_t N, int64_t K, bool fused, const cudaDeviceProp& prop,
                  mxfp4_plan_t* plan);
cudaError_t launch_gemm(const CUtensorMap& tmap_b, const CUtensorMap& tmap_a, const CUtensorMap& tmap_c,
                        const GemmArgs& args, const mxfp4_plan_t& plan, bool fused, bool programmatic,
                        cudaStream_t s);

// ----------------------------------------------------------------------------- multi-layer kernel
// Layers one launch of the multi-layer kernel can run.
constexpr int kMaxChainLayers = 16;

// One layer of a multi-layer launch (device addresses; see chain.cu).
struct ChainLayerArgs {
  const uint8_t* b_sf;       // packed weight scales
  __nv_bfloat16* c;          // output C [M, N]
  const uint8_t* in_sf;      // this layer's activation scale chunks [m_tiles][k_tiles][1 KB]
  const uint32_t* in_done;   // [m_tiles][k_tiles]: readiness of the activation, per K tile
  uint8_t* out_codes;        // next layer's activation codes [M, N/2] (null on the last layer)
  uint8_t* out_sf;           // next layer's activation scale chunks [m_tiles][k_tiles_next][1 KB]
  uint32_t* out_done;        // [m_tiles][k_tiles_next]
  float* partials;           // split-K partials [tiles][splits][block_m][128] fp32
  uint32_t* tickets;         // [tiles]: splits that have stored their partial
  int32_t N, K, k_tiles, kt_per_split, splits, n_tiles, items;
  int32_t in_n_tiles;        // N tiles of the layer producing this one's input (0: the first layer)
  int32_t in_splits;         // K splits of that layer (each split CTA counts its share of a tile)
  int32_t k_tiles_next;
};

struct ChainArgs {
  CUtensorMap wmap[kMaxChainLayers];  // weight codes, per layer
  CUtensorMap amap[kMaxChainLayers];  // activation codes in the workspace, per layer
  ChainLayerArgs layer[kMaxChainLayers];
  const uint16_t* a;         // bf16 A [M, lda] (the first layer's input)
  int64_t lda;
  uint8_t* a_codes;          // the first layer's activation codes [M, K/2]
  uint8_t* a_sf;             // ... and scale chunks
  uint32_t* a_done;          // ... and their readiness counters
  uint32_t* counters;        // every counter of the workspace (zeroed by the last CTA to finish)
  uint32_t* exit_count;
  uint32_t* err;
  uint64_t timeout_ns;
  int32_t n_counters;
  int32_t layers, M, K0, k_tiles0, m_tiles, stages, a_box_rows;
  uint32_t tmem_cols;
  uint32_t a_off, sfw_off, sfa_off, epi_off, bar_off;
  int32_t weights_early;
};

cudaError_t launch_chain(const ChainArgs& args, int block_m, int grid, int smem_bytes, bool programmatic,
                         cudaStream_t s);
// Blocks of the multi-layer kernel that fit on one SM with this shared memory.
int chain_blocks_per_sm(int block_m, int smem_bytes);

cudaError_t read_device_error(cudaStream_t s, uint32_t* code, bool reset);
// The size checks every GEMM entry makes: MXFP4_ERR_INVALID_ARG for
// non-positive sizes or K % 32 != 0, MXFP4_ERR_UNSUPPORTED_SHAPE past the
// kernels' index and grid limits.
mxfp4_status_t check_mnk(int64_t M, int64_t N, int64_t K);
// MXFP4_OK if the current device is an sm_103 GPU, else the status every
// entry returns for it (MXFP4_ERR_UNSUPPORTED_DEVICE or MXFP4_ERR_CUDA).
mxfp4_status_t check_device();
// The fused layer's two-pass route: A quantized into Aq [M, K/2] and As
// [M, K/32] (caller-owned scratch), then the GEMM on the codes.  Every check
// of both launches (device, plan, tensor maps) comes before the first launch;
// an error status means nothing was enqueued.  c_host as for the host entry.
mxfp4_status_t two_pass(const void* A, int64_t lda, const void* Bpacked, void* C, int64_t M, int64_t N, int64_t K,
                        void* Aq, void* As, cudaStream_t s, void* c_host);
// Sets the calling thread's message for mxfp4_last_error_string().
void set_last_error(const char* what);
// Address of the device error word on the current device (nullptr on failure).
uint32_t* device_error_word();

}  // namespace mxfp4
