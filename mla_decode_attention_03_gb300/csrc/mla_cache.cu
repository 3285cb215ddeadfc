// Cache maintenance around MLA decode: writing new tokens into the paged
// latent cache, and copying whole pages (copy_blocks_mla, vLLM PR #12676 "Mem
// align KV caches for CUDA devices").  Both are pure data movement, bound by
// HBM bandwidth: 16-byte vector loads and stores, coalesced per entry / page.
#include <cstdint>

#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kLatentChunks = kDimV / 8;              // 64 x 16 B
constexpr int kEntryChunks = kLatentChunks + 64 / 8;  // + 8 x 16 B of rope

// One warp per token: lanes copy the entry's 72 16-byte chunks.
__global__ void __launch_bounds__(256) mla_write_cache_kernel(const uint4* __restrict__ kv_c, int64_t kv_c_row,
                                                              const uint4* __restrict__ k_pe, int64_t k_pe_row,
                                                              const int64_t* __restrict__ slot_mapping,
                                                              int64_t num_tokens, uint4* __restrict__ kcache,
                                                              int64_t num_slots, int64_t entry_chunks,
                                                              int32_t* __restrict__ status) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= num_tokens) return;
  const int64_t s = slot_mapping[t];
  if (s < 0) return;  // padding token
  if (s >= num_slots) {
    if (lane == 0) atomicExch(status, kStatusBadBlockId);
    return;
  }
  uint4* dst = kcache + s * entry_chunks;
  const uint4* lat = kv_c + t * kv_c_row;
  const uint4* rope = k_pe + t * k_pe_row;
#pragma unroll
  for (int c = lane; c < kEntryChunks; c += 32) dst[c] = (c < kLatentChunks) ? lat[c] : rope[c - kLatentChunks];
}

// Block (pair, layer): copy one page of one layer's cache.
__global__ void __launch_bounds__(256) mla_copy_blocks_kernel(const uint64_t* __restrict__ caches,
                                                              const int64_t* __restrict__ mapping,
                                                              int64_t num_blocks, int64_t page_chunks,
                                                              int32_t* __restrict__ status) {
  const int64_t pair = blockIdx.x;
  const int layer = blockIdx.y;
  const int64_t src = mapping[2 * pair], dst = mapping[2 * pair + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0) atomicExch(status, kStatusBadBlockId);
    return;
  }
  uint4* base = reinterpret_cast<uint4*>(caches[layer]);
  const uint4* from = base + src * page_chunks;
  uint4* to = base + dst * page_chunks;
  for (int64_t c = threadIdx.x; c < page_chunks; c += blockDim.x) to[c] = from[c];
}

}  // namespace

cudaError_t launch_write_cache(const void* kv_c, int64_t kv_c_row_elems, const void* k_pe, int64_t k_pe_row_elems,
                               const int64_t* slot_mapping, int64_t num_tokens, void* kcache, int64_t num_slots,
                               int stride, int32_t* status, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((num_tokens + 7) / 8));
  mla_write_cache_kernel<<<grid, 256, 0, stream>>>(
      static_cast<const uint4*>(kv_c), kv_c_row_elems / 8, static_cast<const uint4*>(k_pe), k_pe_row_elems / 8,
      slot_mapping, num_tokens, static_cast<uint4*>(kcache), num_slots, stride / 8, status);
  return cudaGetLastError();
}

cudaError_t launch_copy_blocks(const uint64_t* caches, int num_layers, const int64_t* mapping, int64_t num_pairs,
                               int64_t num_blocks, int block_size, int stride, int32_t* status,
                               cudaStream_t stream) {
  if (num_pairs == 0 || num_layers == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(num_pairs), static_cast<unsigned>(num_layers));
  mla_copy_blocks_kernel<<<grid, 256, 0, stream>>>(caches, mapping, num_blocks,
                                                   static_cast<int64_t>(block_size) * stride / 8, status);
  return cudaGetLastError();
}

}  // namespace mla
