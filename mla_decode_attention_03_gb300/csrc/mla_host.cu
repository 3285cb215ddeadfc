// Decode from host buffers: the copy-in / decode / copy-out round trip of a
// serving step, pipelined over runs of consecutive sequences (the
// mla_decode_host section of include/mla_decode.h).  Host code only: every
// step of the arithmetic is the decode library's own kernels, enqueued per run
// through the same launch path as mla_decode_with_kvcache.
//
// Streams (more than one run): the caller's stream computes; an internal stream copies inputs in
// (and runs each run's scheduler kernel right behind its copies, so the
// schedule of run k+1 is made while run k decodes); a second internal stream
// copies results out.  Events join them:
//   caller:  rec(start) .. wait(in[k]) decode(k) combine(k) rec(out[k]) .. wait(done)
//   in:      wait(start) wait(done of the previous call) H2D(k) metadata(k) rec(in[k])
//   out:     wait(out[k]) D2H(k) .. rec(done)
// A single run goes entirely on the caller's stream.
// Runs share one split-KV workspace: run k+1's decode kernel is stream-ordered
// after run k's combine on the caller's stream.  Each run has its own
// metadata, because run k+1's schedule is written while run k still reads its
// own.
#include <cuda_runtime.h>

#include <cstdint>
#include <new>

#include "../../include/mla_decode.h"
#include "mla_internal.h"

namespace mla {
// The host-side argument checks of mla_decode_with_kvcache (mla_api.cu):
// MLA_OK or the negative status that call would return.
int32_t check_decode_args(const void* q, int b, int s_q, int h_q, int d, const void* kcache, int64_t num_blocks,
                          int block_size, int h_kv, int stride, const int32_t* block_table,
                          int max_blocks_per_seq, const int32_t* cache_seqlens, int dv,
                          const int32_t* metadata, int num_parts, const int32_t* num_splits,
                          float softmax_scale, int causal, const void* out, const float* lse,
                          const void* workspace, size_t workspace_bytes, const int32_t* status);
}  // namespace mla

struct mla_host_pipeline {
  int device;
  cudaStream_t in, out;
  cudaEvent_t start, done;
  bool has_prev;            // `done` marks the end of an earlier call ...
  cudaStream_t prev_stream; // ... which was made on this caller stream
  cudaEvent_t in_ready[MLA_HOST_MAX_CHUNKS];
  cudaEvent_t out_ready[MLA_HOST_MAX_CHUNKS];
};

namespace {

// Automatic cut: total pages / 2800, rounded, clamped to [1, 3] (measured on the
// benchmark's workloads: b=128 x 64 pages best at 2-3 runs, 128 causal s_q=2
// sequences of ~66 pages best at 3-4, two 1024-page sequences plus 62 short
// ones and 16 short sequences best at 1).
constexpr int kAutoChunkPages = 2800;
constexpr int kAutoMaxChunks = 3;

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Layout {
  size_t q, out, lse, bt, sl, meta, nsplit, ws, ws_bytes, total;
};

Layout layout(int b, int s_q, int h_q, int max_blocks, int parts) {
  const size_t rows = static_cast<size_t>(b) * s_q * h_q;
  Layout L;
  size_t o = 0;
  L.q = o;      o += up256(rows * mla::kDimQK * 2);
  L.out = o;    o += up256(rows * mla::kDimV * 2);
  L.lse = o;    o += up256(rows * sizeof(float));
  L.bt = o;     o += up256(static_cast<size_t>(b) * max_blocks * sizeof(int32_t));
  L.sl = o;     o += up256(static_cast<size_t>(b) * sizeof(int32_t));
  L.meta = o;   o += MLA_HOST_MAX_CHUNKS * up256(static_cast<size_t>(parts) * mla::kMetaInts * sizeof(int32_t));
  L.nsplit = o; o += MLA_HOST_MAX_CHUNKS * up256((static_cast<size_t>(b) + 1) * sizeof(int32_t));
  L.ws = o;
  L.ws_bytes = mla_workspace_bytes(b, s_q, h_q, parts);
  o += L.ws_bytes;
  L.total = o;
  return L;
}

void destroy_members(mla_host_pipeline* p) {
  for (int k = 0; k < MLA_HOST_MAX_CHUNKS; ++k) {
    if (p->in_ready[k]) cudaEventDestroy(p->in_ready[k]);
    if (p->out_ready[k]) cudaEventDestroy(p->out_ready[k]);
  }
  if (p->start) cudaEventDestroy(p->start);
  if (p->done) cudaEventDestroy(p->done);
  if (p->in) cudaStreamDestroy(p->in);
  if (p->out) cudaStreamDestroy(p->out);
}

}  // namespace

extern "C" {

mla_status_t mla_host_pipeline_create(mla_host_pipeline** pipeline) {
  if (!pipeline) return MLA_ERR_INVALID_ARG;
  *pipeline = nullptr;
  mla_host_pipeline* p = new (std::nothrow) mla_host_pipeline{};
  if (!p) return MLA_ERR_CUDA;
  bool ok = cudaGetDevice(&p->device) == cudaSuccess;
  ok = ok && cudaStreamCreateWithFlags(&p->in, cudaStreamNonBlocking) == cudaSuccess;
  ok = ok && cudaStreamCreateWithFlags(&p->out, cudaStreamNonBlocking) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&p->start, cudaEventDisableTiming) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&p->done, cudaEventDisableTiming) == cudaSuccess;
  for (int k = 0; ok && k < MLA_HOST_MAX_CHUNKS; ++k) {
    ok = cudaEventCreateWithFlags(&p->in_ready[k], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->out_ready[k], cudaEventDisableTiming) == cudaSuccess;
  }
  if (!ok) {
    destroy_members(p);
    delete p;
    return MLA_ERR_CUDA;
  }
  *pipeline = p;
  return MLA_OK;
}

mla_status_t mla_host_pipeline_destroy(mla_host_pipeline* pipeline) {
  if (!pipeline) return MLA_OK;
  int prev = 0;
  const bool have_prev = cudaGetDevice(&prev) == cudaSuccess;
  mla_status_t r = MLA_OK;
  if (cudaSetDevice(pipeline->device) != cudaSuccess) r = MLA_ERR_CUDA;
  if (cudaStreamSynchronize(pipeline->in) != cudaSuccess) r = MLA_ERR_CUDA;
  if (cudaStreamSynchronize(pipeline->out) != cudaSuccess) r = MLA_ERR_CUDA;
  destroy_members(pipeline);
  delete pipeline;
  if (have_prev) cudaSetDevice(prev);
  return r;
}

int mla_host_chunks(const int32_t* cache_seqlens, int b, int chunks, int32_t* bounds) {
  if (!cache_seqlens || !bounds || b < 1) return MLA_ERR_INVALID_ARG;
  auto cost = [&](int j) -> int64_t {  // pages of sequence j, plus one
    const int64_t Lj = cache_seqlens[j] > 0 ? cache_seqlens[j] : 0;
    return (Lj + mla::kPage - 1) / mla::kPage + 1;
  };
  int64_t total = 0;
  for (int j = 0; j < b; ++j) total += cost(j);
  const int64_t pages = total - b;
  int n = chunks;
  if (n <= 0) {
    const int64_t a = (pages + kAutoChunkPages / 2) / kAutoChunkPages;
    n = static_cast<int>(a < 1 ? 1 : (a > kAutoMaxChunks ? kAutoMaxChunks : a));
  }
  if (n > MLA_HOST_MAX_CHUNKS) n = MLA_HOST_MAX_CHUNKS;
  if (n > b) n = b;
  // The first and the last run take half a middle run's share of the cost:
  // the first run's copies in and the last run's copies out have no decode to
  // hide behind (measured on the bench workload with 3 runs: 298 -> 287 us).
  // Shares in halves: 1, 2, ..., 2, 1 (two runs: 1, 1).
  const int64_t halves = n <= 2 ? n : 2 * n - 2;
  // i and run track the cost of sequences [0, i)
  bounds[0] = 0;
  int i = 0;
  int64_t run = 0;
  for (int k = 1; k < n; ++k) {
    const int64_t before = n <= 2 ? k : 2 * k - 1;  // halves in runs [0, k)
    const int64_t target = (total * before + halves - 1) / halves;  // ceil(total * before / halves)
    while (i < b && run < target) run += cost(i++);
    int e = i;
    if (e < bounds[k - 1] + 1) e = bounds[k - 1] + 1;  // every run holds a sequence
    if (e > b - (n - k)) e = b - (n - k);               // ... and so do the runs after it
    while (i < e) run += cost(i++);
    while (i > e) run -= cost(--i);
    bounds[k] = e;
  }
  bounds[n] = b;
  return n;
}

size_t mla_host_scratch_bytes(int b, int s_q, int h_q, int max_blocks_per_seq, int num_parts) {
  if (b < 1 || s_q < 1 || h_q < 1 || max_blocks_per_seq < 1 || num_parts < 1) return 0;
  return layout(b, s_q, h_q, max_blocks_per_seq, num_parts).total;
}

mla_status_t mla_decode_host(mla_host_pipeline* pipeline, const void* q, int b, int s_q, int h_q, int d,
                             const void* kcache, int64_t num_blocks, int block_size, int h_kv, int stride,
                             const int32_t* block_table, int max_blocks_per_seq, const int32_t* cache_seqlens,
                             int dv, int num_parts, float softmax_scale, int causal, void* out, float* lse,
                             int chunks, void* scratch, size_t scratch_bytes, int32_t* status,
                             mla_stream_t stream) {
  if (!pipeline || !q || !block_table || !cache_seqlens || !out || !lse || !scratch) return MLA_ERR_INVALID_ARG;
  if (b < 1 || b > mla::kMaxMetadataBatch || s_q < 1 || h_q < 1 || max_blocks_per_seq < 1 || num_parts < 1)
    return MLA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(scratch) & 255u) return MLA_ERR_INVALID_ARG;
  const Layout L = layout(b, s_q, h_q, max_blocks_per_seq, num_parts);
  if (scratch_bytes < L.total) return MLA_ERR_INVALID_ARG;
  // The lengths are on the host here, so the range the device-buffer call can
  // only report (L < 0) or cannot see at all (L above the table's width) is
  // rejected before anything is enqueued.
  const int64_t max_len = static_cast<int64_t>(max_blocks_per_seq) * mla::kPage;
  for (int i = 0; i < b; ++i)
    if (cache_seqlens[i] < 0 || cache_seqlens[i] > max_len) return MLA_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev != pipeline->device) return MLA_ERR_INVALID_ARG;

  char* base = static_cast<char*>(scratch);
  char* q_d = base + L.q;
  char* out_d = base + L.out;
  float* lse_d = reinterpret_cast<float*>(base + L.lse);
  int32_t* bt_d = reinterpret_cast<int32_t*>(base + L.bt);
  int32_t* sl_d = reinterpret_cast<int32_t*>(base + L.sl);
  void* ws = base + L.ws;
  const size_t meta_stride = up256(static_cast<size_t>(num_parts) * mla::kMetaInts * sizeof(int32_t));
  const size_t nsplit_stride = up256((static_cast<size_t>(b) + 1) * sizeof(int32_t));
  auto meta_of = [&](int k) { return reinterpret_cast<int32_t*>(base + L.meta + k * meta_stride); };
  auto nsplit_of = [&](int k) { return reinterpret_cast<int32_t*>(base + L.nsplit + k * nsplit_stride); };

  // every host-side check of the per-run decode calls, on the whole batch, before anything is enqueued
  const mla_status_t chk = mla::check_decode_args(
      q_d, b, s_q, h_q, d, kcache, num_blocks, block_size, h_kv, stride, bt_d, max_blocks_per_seq, sl_d, dv,
      meta_of(0), num_parts, nsplit_of(0), softmax_scale, causal, out_d, lse_d, ws, L.ws_bytes, status);
  if (chk != MLA_OK) return chk;

  int32_t bounds[MLA_HOST_MAX_CHUNKS + 1];
  const int n = mla_host_chunks(cache_seqlens, b, chunks, bounds);
  if (n < 1) return MLA_ERR_INVALID_ARG;

  const size_t q_row = static_cast<size_t>(s_q) * h_q * mla::kDimQK * 2;  // bytes per sequence
  const size_t o_row = static_cast<size_t>(s_q) * h_q * mla::kDimV * 2;
  const size_t l_row = static_cast<size_t>(s_q) * h_q * sizeof(float);
  const size_t bt_row = static_cast<size_t>(max_blocks_per_seq) * sizeof(int32_t);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  mla_host_pipeline* P = pipeline;
  const char* qh = static_cast<const char*>(q);
  const char* bth = reinterpret_cast<const char*>(block_table);
  char* oh = static_cast<char*>(out);
  char* lh = reinterpret_cast<char*>(lse);

#define MLA_CUDA(x)                                \
  do {                                             \
    if ((x) != cudaSuccess) return MLA_ERR_CUDA;   \
  } while (0)

  // One run needs no overlap: copies, schedule, decode and copies back all go
  // on the caller's stream, without the event hops between streams.
  const bool split = n > 1;
  cudaStream_t in_s = split ? P->in : cs;
  cudaStream_t out_s = split ? P->out : cs;
  auto enqueue = [&]() -> mla_status_t {
    if (split) {
      MLA_CUDA(cudaEventRecord(P->start, cs));
      MLA_CUDA(cudaStreamWaitEvent(P->in, P->start, 0));
      MLA_CUDA(cudaStreamWaitEvent(P->out, P->start, 0));
    }
    // the previous call on this pipeline has finished (implied by stream order on the same caller stream)
    if (P->has_prev && P->prev_stream != cs) MLA_CUDA(cudaStreamWaitEvent(in_s, P->done, 0));
    for (int k = 0; k < n; ++k) {
      const int i0 = bounds[k], bk = bounds[k + 1] - bounds[k];
      MLA_CUDA(cudaMemcpyAsync(q_d + i0 * q_row, qh + i0 * q_row, bk * q_row, cudaMemcpyHostToDevice, in_s));
      MLA_CUDA(cudaMemcpyAsync(reinterpret_cast<char*>(bt_d) + i0 * bt_row, bth + i0 * bt_row, bk * bt_row,
                               cudaMemcpyHostToDevice, in_s));
      MLA_CUDA(cudaMemcpyAsync(sl_d + i0, cache_seqlens + i0, bk * sizeof(int32_t), cudaMemcpyHostToDevice, in_s));
      const mla_status_t r = mla_get_metadata(sl_d + i0, bk, num_parts, meta_of(k), nsplit_of(k), status, in_s);
      if (r != MLA_OK) return r;
      if (split) MLA_CUDA(cudaEventRecord(P->in_ready[k], in_s));
    }
    for (int k = 0; k < n; ++k) {
      const int i0 = bounds[k], bk = bounds[k + 1] - bounds[k];
      if (split) MLA_CUDA(cudaStreamWaitEvent(cs, P->in_ready[k], 0));
      const mla_status_t r = mla_decode_with_kvcache(
          q_d + i0 * q_row, bk, s_q, h_q, d, kcache, num_blocks, block_size, h_kv, stride,
          reinterpret_cast<const int32_t*>(reinterpret_cast<const char*>(bt_d) + i0 * bt_row), max_blocks_per_seq,
          sl_d + i0, dv, meta_of(k), num_parts, nsplit_of(k), softmax_scale, causal, out_d + i0 * o_row,
          reinterpret_cast<float*>(reinterpret_cast<char*>(lse_d) + i0 * l_row), ws, L.ws_bytes, status, stream);
      if (r != MLA_OK) return r;
      if (split) {
        MLA_CUDA(cudaEventRecord(P->out_ready[k], cs));
        MLA_CUDA(cudaStreamWaitEvent(P->out, P->out_ready[k], 0));
      }
      MLA_CUDA(cudaMemcpyAsync(oh + i0 * o_row, out_d + i0 * o_row, bk * o_row, cudaMemcpyDeviceToHost, out_s));
      MLA_CUDA(cudaMemcpyAsync(lh + i0 * l_row, reinterpret_cast<char*>(lse_d) + i0 * l_row, bk * l_row,
                               cudaMemcpyDeviceToHost, out_s));
    }
    MLA_CUDA(cudaEventRecord(P->done, out_s));
    if (split) MLA_CUDA(cudaStreamWaitEvent(cs, P->done, 0));
    return MLA_OK;
  };
  const mla_status_t r = enqueue();
  if (r != MLA_OK && split) {
    // Something failed after work may already be queued on the side streams:
    // join them into the caller's stream anyway (best effort), so that no copy
    // of this call can still be writing the caller's buffers after its stream
    // has passed this point, and the next call waits for them.
    if (cudaEventRecord(P->done, in_s) == cudaSuccess) cudaStreamWaitEvent(out_s, P->done, 0);
    if (cudaEventRecord(P->done, out_s) == cudaSuccess) cudaStreamWaitEvent(cs, P->done, 0);
  }
  P->has_prev = true;
  P->prev_stream = cs;
#undef MLA_CUDA
  return r;
}

}  // extern "C"
