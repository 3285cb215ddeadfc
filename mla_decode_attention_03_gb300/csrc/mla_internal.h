// Internal interface between the C-ABI host code and the CUDA kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace mla {

constexpr int kDimQK = 576;     // latent 512 + rope 64
constexpr int kDimV = 512;      // value = leading 512 latent dims
constexpr int kPage = 64;       // tokens per cache page
constexpr int kRowsPerTile = 128;
constexpr int kSmallTileRows = 16;  // tiles of at most this many rows take the one-CTA kernel
constexpr int kMetaInts = 8;    // ints per scheduler part
constexpr int kSegmentCost = 6; // fixed scheduler cost of one (sequence, part) segment, in pages (measured: 2, 4, 6, 8, 12 -> 6 best)
constexpr int kMinPartCost = 4;   // smallest part, in cost units (independent of kSegmentCost)
constexpr int kMaxMetadataBatch = 16384;  // sequences the scheduler stages in shared memory

// Device-side status codes (written to the caller's status word).
enum : int32_t {
  kStatusOk = 0,
  kStatusBadBlockId = -5,
  kStatusTimeout = -6,
  kStatusBadSeqlen = -7,
};

struct DecodeParams {
  const void* q;                 // bf16 [b, s_q, h_q, 576]
  const int32_t* block_table;    // [b, max_blocks]
  const int32_t* cache_seqlens;  // [b]
  const int32_t* metadata;       // [num_parts, kMetaInts]
  const int32_t* num_splits;     // [b + 1] prefix sums
  void* out;                     // bf16 [b, s_q, h_q, 512]
  float* lse;                    // [b, h_q, s_q]
  void* ws_o;                    // fp32 [slots, s_q*h_q, 512]: normalised partial outputs
  float* ws_lse;                 // [slots, s_q*h_q]
  int32_t* status;
  int64_t num_blocks;
  int b, s_q, h_q, h_kv;
  int heads_per_kv;   // h_q / h_kv
  int q_per_tile;     // query positions per row tile
  int rows_per_tile;  // heads_per_kv * q_per_tile  (<= 128)
  int max_blocks;
  int causal;
  float scale_log2;   // softmax_scale * log2(e)
  int stall_test;     // diagnostic: the TMA producer first waits on a barrier nothing completes
};

struct CombineParams {
  const int32_t* num_splits;
  const void* ws_o;              // fp32 partial outputs
  const float* ws_lse;
  void* out;
  float* lse;
  int b, s_q, h_q;
  int num_parts;                 // the schedule's part count (host side: picks the kernel shape)
};

int decode_smem_bytes();
cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& q_rope, const CUtensorMap& k_lat,
                          const CUtensorMap& k_rope, int num_parts, int row_tiles, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);
cudaError_t launch_metadata(const int32_t* cache_seqlens, int b, int num_parts, int32_t* metadata,
                            int32_t* num_splits, int32_t* status, cudaStream_t stream);
cudaError_t decode_max_active_clusters(int* clusters);
// One CTA per (part, KV head) for shapes with s_q * heads_per_kv <= kSmallTileRows.
int decode_small_smem_bytes();
cudaError_t launch_decode_small(const DecodeParams& p, const CUtensorMap& q_full, const CUtensorMap& k_lat, int num_parts,
                                cudaStream_t stream);
cudaError_t decode_small_max_ctas(int* ctas);
cudaError_t launch_write_cache(const void* kv_c, int64_t kv_c_row_elems, const void* k_pe, int64_t k_pe_row_elems,
                               const int64_t* slot_mapping, int64_t num_tokens, void* kcache, int64_t num_slots,
                               int stride, int32_t* status, cudaStream_t stream);
cudaError_t launch_copy_blocks(const uint64_t* caches, int num_layers, const int64_t* mapping, int64_t num_pairs,
                               int64_t num_blocks, int block_size, int stride, int32_t* status,
                               cudaStream_t stream);

}  // namespace mla
