// Host side of the C ABI declared in include/mla_decode.h: argument checks,
// TMA tensor maps and kernel launches.  No allocation, no synchronisation.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/mla_decode.h"
#include "mla_internal.h"

namespace {

using mla::kDimQK;
using mla::kDimV;
using mla::kPage;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Shape {
  int heads_per_kv, q_per_tile, rows_per_tile, row_tiles;
};

Shape tile_shape(int s_q, int h_q, int h_kv) {
  Shape s;
  s.heads_per_kv = h_q / h_kv;
  s.q_per_tile = mla::kRowsPerTile / s.heads_per_kv;
  if (s.q_per_tile > s_q) s.q_per_tile = s_q;
  if (s.q_per_tile < 1) s.q_per_tile = 1;
  s.rows_per_tile = s.heads_per_kv * s.q_per_tile;
  s.row_tiles = (s_q + s.q_per_tile - 1) / s.q_per_tile;
  return s;
}

// Tiles of at most 16 rows (one query position x up to 16 heads per KV head,
// or a few positions x fewer heads) run on the one-CTA kernel.
bool small_tile(int s_q, int h_q, int h_kv) {
  return static_cast<int64_t>(s_q) * (h_q / h_kv) <= mla::kSmallTileRows;
}

size_t workspace_o_bytes(int b, int s_q, int h_q, int num_parts) {
  const size_t slots = static_cast<size_t>(b) + static_cast<size_t>(num_parts);
  const size_t bytes = slots * static_cast<size_t>(s_q) * h_q * kDimV * 4;  // fp32 partials
  return (bytes + 255) & ~static_cast<size_t>(255);
}

mla_status_t encode(CUtensorMap* map, int rank, void* base, const cuuint64_t* dims,
                    const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz) {
  auto enc = tensor_map_encoder();
  if (!enc) return MLA_ERR_CUDA;
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, base, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* mla_status_string(mla_status_t s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: argument outside the accepted range";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: shape not supported (d=576, dv=512, block_size=64, h_q/h_kv<=128)";
    case MLA_ERR_ALIGNMENT: return "MLA_ERR_ALIGNMENT: pointer or stride not 16-byte aligned";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: a CUDA call failed";
    case MLA_ERR_BAD_BLOCK_ID: return "MLA_ERR_BAD_BLOCK_ID: block_table entry outside [0, num_blocks)";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a decode pipeline wait gave up";
    case MLA_ERR_BAD_SEQLEN: return "MLA_ERR_BAD_SEQLEN: negative cache_seqlens entry";
    case MLA_ERR_SCRATCH_TOO_SMALL: return "MLA_ERR_SCRATCH_TOO_SMALL: shape needs more split-KV scratch than the library's built-in 64 MiB";
    default: return "MLA: unknown status";
  }
}

int mla_num_parts(int s_q, int h_q, int h_kv, int device) {
  if (s_q < 1 || h_q < 1 || h_kv < 1 || h_q % h_kv != 0) return MLA_ERR_INVALID_ARG;
  if (h_q / h_kv > mla::kRowsPerTile) return MLA_ERR_UNSUPPORTED;
  static std::mutex mu;
  static int cached[64][2];  // resident 2-CTA clusters of the 128-row kernel, CTAs of the 16-row kernel
  static bool have[64] = {false};
  if (device < 0 || device >= 64) return MLA_ERR_INVALID_ARG;
  const bool small = small_tile(s_q, h_q, h_kv);
  int units = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!have[device]) {
      int prev = 0;
      if (cudaGetDevice(&prev) != cudaSuccess) return MLA_ERR_CUDA;
      if (cudaSetDevice(device) != cudaSuccess) return MLA_ERR_CUDA;
      int c = 0, k = 0;
      cudaError_t e = mla::decode_max_active_clusters(&c);
      if (e == cudaSuccess) e = mla::decode_small_max_ctas(&k);
      cudaSetDevice(prev);
      if (e != cudaSuccess || c < 1 || k < 1) return MLA_ERR_CUDA;
      cached[device][0] = c;
      cached[device][1] = k;
      have[device] = true;
    }
    units = cached[device][small ? 1 : 0];
  }
  const Shape s = tile_shape(s_q, h_q, h_kv);
  int parts = small ? units / h_kv : units / (s.row_tiles * h_kv);
  return parts < 1 ? 1 : parts;
}

size_t mla_metadata_ints(int num_parts) {
  return num_parts > 0 ? static_cast<size_t>(num_parts) * mla::kMetaInts : 0;
}

size_t mla_workspace_bytes(int b, int s_q, int h_q, int num_parts) {
  if (b < 1 || s_q < 1 || h_q < 1 || num_parts < 1) return 0;
  const size_t slots = static_cast<size_t>(b) + static_cast<size_t>(num_parts);
  const size_t lse = slots * static_cast<size_t>(s_q) * h_q * sizeof(float);
  return workspace_o_bytes(b, s_q, h_q, num_parts) + ((lse + 255) & ~static_cast<size_t>(255));
}

mla_status_t mla_get_metadata(const int32_t* cache_seqlens, int b, int num_parts, int32_t* metadata,
                              int32_t* num_splits, int32_t* status, mla_stream_t stream) {
  if (!cache_seqlens || !metadata || !num_splits || !status) return MLA_ERR_INVALID_ARG;
  if (b < 1 || b > mla::kMaxMetadataBatch || num_parts < 1) return MLA_ERR_INVALID_ARG;
  cudaError_t e = mla::launch_metadata(cache_seqlens, b, num_parts, metadata, num_splits, status,
                                       reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // extern "C"

namespace mla {

int32_t check_decode_args(const void* q, int b, int s_q, int h_q, int d, const void* kcache, int64_t num_blocks,
                          int block_size, int h_kv, int stride, const int32_t* block_table,
                          int max_blocks_per_seq, const int32_t* cache_seqlens, int dv,
                          const int32_t* metadata, int num_parts, const int32_t* num_splits,
                          float softmax_scale, int causal, const void* out, const float* lse,
                          const void* workspace, size_t workspace_bytes, const int32_t* status) {
  if (!q || !kcache || !block_table || !cache_seqlens || !metadata || !num_splits || !out || !lse ||
      !workspace || !status)
    return MLA_ERR_INVALID_ARG;
  if (b < 1 || s_q < 1 || h_q < 1 || h_kv < 1 || num_blocks < 1 || max_blocks_per_seq < 1 ||
      num_parts < 1 || (causal != 0 && causal != 1) || !std::isfinite(softmax_scale) || !(softmax_scale > 0.f))
    return MLA_ERR_INVALID_ARG;
  if (h_q % h_kv != 0) return MLA_ERR_INVALID_ARG;
  if (d != kDimQK || dv != kDimV || block_size != kPage || h_q / h_kv > mla::kRowsPerTile)
    return MLA_ERR_UNSUPPORTED;
  if (stride < kDimQK) return MLA_ERR_INVALID_ARG;
  if (stride % 8 != 0) return MLA_ERR_ALIGNMENT;
  if (num_blocks * kPage * static_cast<int64_t>(h_kv) >= (static_cast<int64_t>(1) << 31))
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(out) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return MLA_ERR_ALIGNMENT;
  if (workspace_bytes < mla_workspace_bytes(b, s_q, h_q, num_parts)) return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(s_q) * h_q > 4 * 65535) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

}  // namespace mla

namespace {

mla_status_t decode_impl(const void* q, int b, int s_q, int h_q, int d, const void* kcache,
                         int64_t num_blocks, int block_size, int h_kv, int stride,
                         const int32_t* block_table, int max_blocks_per_seq,
                         const int32_t* cache_seqlens, int dv, const int32_t* metadata, int num_parts,
                         const int32_t* num_splits, float softmax_scale, int causal, void* out,
                         float* lse, void* workspace, size_t workspace_bytes, int32_t* status,
                         mla_stream_t stream, bool with_combine, bool stall_test = false) {
  const mla_status_t chk = mla::check_decode_args(
      q, b, s_q, h_q, d, kcache, num_blocks, block_size, h_kv, stride, block_table, max_blocks_per_seq,
      cache_seqlens, dv, metadata, num_parts, num_splits, softmax_scale, causal, out, lse, workspace,
      workspace_bytes, status);
  if (chk != MLA_OK) return chk;

  const Shape s = tile_shape(s_q, h_q, h_kv);
  const bool small = small_tile(s_q, h_q, h_kv);
  CUtensorMap q_rope, k_lat, k_rope;
  const cuuint64_t qrow = static_cast<cuuint64_t>(kDimQK) * 2;
  const cuuint64_t entry = static_cast<cuuint64_t>(stride) * 2;
  if (small) {
    // 16-row kernel: views whose two innermost dimensions are (64 dims, 9
    // slices of 64), so that one copy moves a segment's Q (all its rows) or
    // a page (all 64 tokens) as 128-byte (row, slice) rows, 128B swizzle
    cuuint64_t qdims[5] = {64, kDimQK / 64, static_cast<cuuint64_t>(h_q), static_cast<cuuint64_t>(s_q),
                           static_cast<cuuint64_t>(b)};
    cuuint64_t qstrides[4] = {128, qrow, qrow * h_q, qrow * h_q * s_q};
    cuuint32_t qbox[5] = {64, kDimQK / 64, static_cast<cuuint32_t>(s.heads_per_kv),
                          static_cast<cuuint32_t>(s_q), 1};
    mla_status_t r = encode(&q_rope, 5, const_cast<void*>(q), qdims, qstrides, qbox, CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != MLA_OK) return r;
    cuuint64_t kdims[4] = {64, kDimQK / 64, static_cast<cuuint64_t>(h_kv), static_cast<cuuint64_t>(num_blocks) * kPage};
    cuuint64_t kstrides[3] = {128, entry, entry * h_kv};
    cuuint32_t kbox[4] = {64, kDimQK / 64, 1, static_cast<cuuint32_t>(kPage)};
    r = encode(&k_lat, 4, const_cast<void*>(kcache), kdims, kstrides, kbox, CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != MLA_OK) return r;
  } else {
    {
      // the 32 rope dims of each CTA's Q columns; its latent dims are read by the kernel's threads
      cuuint64_t dims[4] = {static_cast<cuuint64_t>(kDimQK), static_cast<cuuint64_t>(h_q),
                            static_cast<cuuint64_t>(s_q), static_cast<cuuint64_t>(b)};
      cuuint64_t strides[3] = {qrow, qrow * h_q, qrow * h_q * s_q};
      cuuint32_t box[4] = {32, static_cast<cuuint32_t>(s.heads_per_kv), static_cast<cuuint32_t>(s.q_per_tile), 1};
      mla_status_t r = encode(&q_rope, 4, const_cast<void*>(q), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
      if (r != MLA_OK) return r;
    }
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDimQK), static_cast<cuuint64_t>(h_kv),
                          static_cast<cuuint64_t>(num_blocks) * kPage};
    cuuint64_t strides[2] = {entry, entry * h_kv};
    cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kPage)};
    mla_status_t r = encode(&k_lat, 3, const_cast<void*>(kcache), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != MLA_OK) return r;
    box[0] = 32;
    r = encode(&k_rope, 3, const_cast<void*>(kcache), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
    if (r != MLA_OK) return r;
  }

  void* ws_o = workspace;
  float* ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                           workspace_o_bytes(b, s_q, h_q, num_parts));
  mla::DecodeParams p;
  p.q = q;
  p.block_table = block_table;
  p.cache_seqlens = cache_seqlens;
  p.metadata = metadata;
  p.num_splits = num_splits;
  p.out = out;
  p.lse = lse;
  p.ws_o = ws_o;
  p.ws_lse = ws_lse;
  p.status = status;
  p.num_blocks = num_blocks;
  p.b = b;
  p.s_q = s_q;
  p.h_q = h_q;
  p.h_kv = h_kv;
  p.heads_per_kv = s.heads_per_kv;
  p.q_per_tile = s.q_per_tile;
  p.rows_per_tile = s.rows_per_tile;
  p.max_blocks = max_blocks_per_seq;
  p.causal = causal;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.stall_test = stall_test ? 1 : 0;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = small ? mla::launch_decode_small(p, q_rope, k_lat, num_parts, st)
                       : mla::launch_decode(p, q_rope, k_lat, k_rope, num_parts, s.row_tiles, st);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  if (!with_combine) return MLA_OK;
  return mla_combine_splits(num_splits, b, s_q, h_q, workspace, num_parts, out, lse, stream);
}

}  // namespace

extern "C" {

mla_status_t mla_decode_with_kvcache(const void* q, int b, int s_q, int h_q, int d, const void* kcache,
                                     int64_t num_blocks, int block_size, int h_kv, int stride,
                                     const int32_t* block_table, int max_blocks_per_seq,
                                     const int32_t* cache_seqlens, int dv, const int32_t* metadata,
                                     int num_parts, const int32_t* num_splits, float softmax_scale,
                                     int causal, void* out, float* lse, void* workspace,
                                     size_t workspace_bytes, int32_t* status, mla_stream_t stream) {
  return decode_impl(q, b, s_q, h_q, d, kcache, num_blocks, block_size, h_kv, stride, block_table,
                     max_blocks_per_seq, cache_seqlens, dv, metadata, num_parts, num_splits,
                     softmax_scale, causal, out, lse, workspace, workspace_bytes, status, stream, true);
}

mla_status_t mla_decode_splitkv(const void* q, int b, int s_q, int h_q, int d, const void* kcache,
                                int64_t num_blocks, int block_size, int h_kv, int stride,
                                const int32_t* block_table, int max_blocks_per_seq,
                                const int32_t* cache_seqlens, int dv, const int32_t* metadata,
                                int num_parts, const int32_t* num_splits, float softmax_scale,
                                int causal, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, int32_t* status, mla_stream_t stream) {
  return decode_impl(q, b, s_q, h_q, d, kcache, num_blocks, block_size, h_kv, stride, block_table,
                     max_blocks_per_seq, cache_seqlens, dv, metadata, num_parts, num_splits,
                     softmax_scale, causal, out, lse, workspace, workspace_bytes, status, stream, false);
}

mla_status_t mla_selftest_wait_timeout(const void* q, int b, int s_q, int h_q, int d, const void* kcache,
                                       int64_t num_blocks, int block_size, int h_kv, int stride,
                                       const int32_t* block_table, int max_blocks_per_seq,
                                       const int32_t* cache_seqlens, int dv, const int32_t* metadata,
                                       int num_parts, const int32_t* num_splits, float softmax_scale, int causal,
                                       void* out, float* lse, void* workspace, size_t workspace_bytes,
                                       int32_t* status, mla_stream_t stream) {
  return decode_impl(q, b, s_q, h_q, d, kcache, num_blocks, block_size, h_kv, stride, block_table,
                     max_blocks_per_seq, cache_seqlens, dv, metadata, num_parts, num_splits, softmax_scale,
                     causal, out, lse, workspace, workspace_bytes, status, stream, true, true);
}

mla_status_t mla_write_cache(const void* kv_c, int64_t kv_c_row_stride, const void* k_pe, int64_t k_pe_row_stride,
                             const int64_t* slot_mapping, int64_t num_tokens, void* kcache, int64_t num_blocks,
                             int block_size, int stride, int32_t* status, mla_stream_t stream) {
  if (num_tokens < 0 || num_blocks < 1 || !kcache || !status) return MLA_ERR_INVALID_ARG;
  if (num_tokens > 0 && (!kv_c || !k_pe || !slot_mapping)) return MLA_ERR_INVALID_ARG;
  if (block_size != kPage) return MLA_ERR_UNSUPPORTED;
  if (stride < kDimQK || kv_c_row_stride < kDimV || k_pe_row_stride < kDimQK - kDimV) return MLA_ERR_INVALID_ARG;
  if (stride % 8 || kv_c_row_stride % 8 || k_pe_row_stride % 8) return MLA_ERR_ALIGNMENT;
  if ((num_tokens > 0 && (!aligned16(kv_c) || !aligned16(k_pe))) || !aligned16(kcache)) return MLA_ERR_ALIGNMENT;
  if ((num_tokens + 7) / 8 > 0x7fffffff) return MLA_ERR_INVALID_ARG;
  return mla::launch_write_cache(kv_c, kv_c_row_stride, k_pe, k_pe_row_stride, slot_mapping, num_tokens, kcache,
                                 num_blocks * kPage, stride, status, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

mla_status_t mla_copy_blocks(const uint64_t* kcaches, int num_layers, const int64_t* block_mapping,
                             int64_t num_pairs, int64_t num_blocks, int block_size, int stride, int32_t* status,
                             mla_stream_t stream) {
  if (num_layers < 0 || num_layers > 65535 || num_pairs < 0 || num_pairs > 0x7fffffff || num_blocks < 1 || !status)
    return MLA_ERR_INVALID_ARG;
  if (num_layers > 0 && num_pairs > 0 && (!kcaches || !block_mapping)) return MLA_ERR_INVALID_ARG;
  if (block_size != kPage) return MLA_ERR_UNSUPPORTED;
  if (stride < kDimQK) return MLA_ERR_INVALID_ARG;
  if (stride % 8) return MLA_ERR_ALIGNMENT;
  return mla::launch_copy_blocks(kcaches, num_layers, block_mapping, num_pairs, num_blocks, block_size, stride,
                                 status, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

mla_status_t mla_combine_splits(const int32_t* num_splits, int b, int s_q, int h_q,
                                const void* workspace, int num_parts, void* out, float* lse,
                                mla_stream_t stream) {
  if (!num_splits || !workspace || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (b < 1 || s_q < 1 || h_q < 1 || num_parts < 1) return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(s_q) * h_q > 4 * 65535) return MLA_ERR_UNSUPPORTED;
  if (!aligned16(workspace) || !aligned16(out) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return MLA_ERR_ALIGNMENT;
  mla::CombineParams c;
  c.num_splits = num_splits;
  c.ws_o = workspace;
  c.ws_lse = reinterpret_cast<const float*>(static_cast<const char*>(workspace) +
                                            workspace_o_bytes(b, s_q, h_q, num_parts));
  c.out = out;
  c.lse = lse;
  c.b = b;
  c.s_q = s_q;
  c.h_q = h_q;
  c.num_parts = num_parts;
  return mla::launch_combine(c, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? MLA_OK
                                                                                         : MLA_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant.  The split-KV scratch lives in this file-scope
// device array instead of a caller-provided workspace.  Host code may not use
// the array's name as a device address (on the host it only stands for the
// symbol), so its address is looked up once per device with that device
// current, and that address is what the kernels receive.
namespace {

static __device__ __align__(256) unsigned char g_static_workspace[MLA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

mla_status_t static_workspace(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return MLA_ERR_CUDA;
    g_static_ptr[dev] = p;
  }
  *ptr = g_static_ptr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" mla_status_t mla_decode_with_kvcache_static(
    const void* q, int b, int s_q, int h_q, int d, const void* kcache, int64_t num_blocks, int block_size,
    int h_kv, int stride, const int32_t* block_table, int max_blocks_per_seq, const int32_t* cache_seqlens,
    int dv, const int32_t* metadata, int num_parts, const int32_t* num_splits, float softmax_scale,
    int causal, void* out, float* lse, int32_t* status, mla_stream_t stream) {
  const size_t need = mla_workspace_bytes(b, s_q, h_q, num_parts);
  if (need == 0) return MLA_ERR_INVALID_ARG;
  if (need > MLA_STATIC_WORKSPACE_BYTES) return MLA_ERR_SCRATCH_TOO_SMALL;
  void* ws = nullptr;
  const mla_status_t r = static_workspace(&ws);
  if (r != MLA_OK) return r;
  return decode_impl(q, b, s_q, h_q, d, kcache, num_blocks, block_size, h_kv, stride, block_table,
                     max_blocks_per_seq, cache_seqlens, dv, metadata, num_parts, num_splits,
                     softmax_scale, causal, out, lse, ws, MLA_STATIC_WORKSPACE_BYTES, status, stream, true);
}
