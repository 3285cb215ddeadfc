// Split-KV scheduling metadata and the log-sum-exp combine.
//
// Flash-Decoding (as the Hacker News thread on the FlashMLA release describes
// it) adds the KV length as a parallel dimension: a long sequence is cut into
// pieces that run on different SMs, and the partial results are merged using
// their log-sum-exps.  FlashMLA's get_mla_metadata, which vLLM's
// FlashMLAMetadataBuilder calls once per decode step (PAI tutorial, section 2),
// computes that cut; this file holds this library's own version of it and the
// merge kernel.
#include <cuda_bf16.h>

#include "mla_internal.h"

namespace mla {
namespace {

// Greedy balanced cut of the (sequence, page) order into num_parts contiguous
// parts.  Every (sequence, part) segment costs its pages plus kSegmentCost;
// each part takes about (total + split overheads)/num_parts.  Output per part:
//   meta[0] = first sequence, meta[1] = first page in it,
//   meta[2] = last sequence,  meta[3] = end page (exclusive) in the last one,
//   meta[4] = split index of the first segment within its sequence.
// An empty part has meta[0] > meta[2].  num_splits[b+1] is the exclusive
// prefix sum of the number of segments of each sequence.
__global__ void __launch_bounds__(256) mla_metadata_kernel(const int32_t* __restrict__ seqlens, int b,
                                                           int num_parts, int32_t* __restrict__ meta,
                                                           int32_t* __restrict__ num_splits,
                                                           int32_t* __restrict__ status) {
  extern __shared__ int32_t sh[];  // [0, b): pages per sequence; [b, 2b): segments per sequence
  int32_t* pages = sh;
  int32_t* segs = sh + b;
  for (int i = threadIdx.x; i < b; i += blockDim.x) {
    const int L = seqlens[i];
    if (L < 0) atomicExch(status, kStatusBadSeqlen);
    pages[i] = L > 0 ? (L + kPage - 1) / kPage : 0;
    segs[i] = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    long long total = 0;
    for (int i = 0; i < b; ++i)
      if (pages[i] > 0) total += pages[i] + kSegmentCost;
    // Each part boundary that falls inside a sequence adds one more segment
    // (and its fixed cost); budget for up to num_parts-1 of them.
    const long long estimate = total + static_cast<long long>(kSegmentCost) * (num_parts - 1);
    long long per_part = (estimate + num_parts - 1) / num_parts;
    if (per_part < kSegmentCost + kMinPartPages) per_part = kSegmentCost + kMinPartPages;

    // Part q ends near cumulative cost (q+1)*per_part, so a part that stops a
    // little short does not push the shortfall onto the last part.
    long long consumed = 0;
    int i = 0, p = 0, k = 0, part = 0;
    while (i < b && pages[i] == 0) ++i;
    for (; part < num_parts && i < b; ++part) {
      int32_t* m = meta + part * kMetaInts;
      m[0] = i;
      m[1] = p;
      m[4] = k;
      m[5] = m[6] = m[7] = 0;
      const bool last_part = (part == num_parts - 1);
      long long budget = (part + 1) * per_part - consumed;
      int last_i = i, last_end = p;
      while (i < b) {
        if (pages[i] == 0) {
          ++i;
          continue;
        }
        if (!last_part && budget < kSegmentCost + 1) break;
        const long long need = kSegmentCost + (pages[i] - p);
        if (last_part || need <= budget) {
          budget -= need;
          consumed += need;
          segs[i] = k + 1;
          last_i = i;
          last_end = pages[i];
          ++i;
          p = 0;
          k = 0;
        } else {
          const int take = static_cast<int>(budget - kSegmentCost);  // >= 1
          consumed += budget;
          segs[i] = k + 1;
          last_i = i;
          p += take;
          last_end = p;
          ++k;
          break;
        }
      }
      if (last_end == m[1] && last_i == m[0]) {
        m[0] = 1;  // nothing placed: empty part
        m[2] = 0;
      } else {
        m[2] = last_i;
      }
      m[3] = last_end;
      while (i < b && pages[i] == 0) ++i;
    }
    for (; part < num_parts; ++part) {
      int32_t* m = meta + part * kMetaInts;
      m[0] = 1;
      m[1] = 0;
      m[2] = 0;
      m[3] = 0;
      m[4] = m[5] = m[6] = m[7] = 0;
    }
    int acc = 0;
    num_splits[0] = 0;
    for (int s = 0; s < b; ++s) {
      acc += segs[s];
      num_splits[s + 1] = acc;
    }
  }
}

// One warp per (sequence, query row).  Sequences with a single split were
// written directly by the decode kernel; sequences with none (length 0) get
// out = 0 and lse = -inf.
__global__ void __launch_bounds__(128) mla_combine_kernel(const CombineParams P) {
  const int i = blockIdx.x;
  const int rows = P.s_q * P.h_q;
  const int row = blockIdx.y * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int s0 = P.num_splits[i];
  const int ns = P.num_splits[i + 1] - s0;
  if (ns == 1) return;
  const int j = row / P.h_q, h = row - (row / P.h_q) * P.h_q;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(P.out) + (static_cast<int64_t>(i) * rows + row) * kDimV;
  float* lse_out = P.lse + (static_cast<int64_t>(i) * P.h_q + h) * P.s_q + j;

  float mx = -INFINITY;
  for (int k = lane; k < ns; k += 32) mx = fmaxf(mx, P.ws_lse[static_cast<int64_t>(s0 + k) * rows + row]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));

  float acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.f;
  float lse = -INFINITY;
  if (ns > 0 && mx != -INFINITY) {
    float sum = 0.f;
    for (int k = lane; k < ns; k += 32) sum += expf(P.ws_lse[static_cast<int64_t>(s0 + k) * rows + row] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    lse = mx + logf(sum);
    for (int k = 0; k < ns; ++k) {
      const int64_t r = static_cast<int64_t>(s0 + k) * rows + row;
      const float wgt = expf(P.ws_lse[r] - lse);
      const float4* src = reinterpret_cast<const float4*>(P.ws_o + r * kDimV) + lane * 4;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = src[q];
        acc[4 * q + 0] += wgt * v.x;
        acc[4 * q + 1] += wgt * v.y;
        acc[4 * q + 2] += wgt * v.z;
        acc[4 * q + 3] += wgt * v.w;
      }
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(out) + lane * 2;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    __nv_bfloat162 a = __floats2bfloat162_rn(acc[8 * q + 0], acc[8 * q + 1]);
    __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[8 * q + 2], acc[8 * q + 3]);
    __nv_bfloat162 c = __floats2bfloat162_rn(acc[8 * q + 4], acc[8 * q + 5]);
    __nv_bfloat162 d = __floats2bfloat162_rn(acc[8 * q + 6], acc[8 * q + 7]);
    uint4 v;
    v.x = *reinterpret_cast<uint32_t*>(&a);
    v.y = *reinterpret_cast<uint32_t*>(&b2);
    v.z = *reinterpret_cast<uint32_t*>(&c);
    v.w = *reinterpret_cast<uint32_t*>(&d);
    dst[q] = v;
  }
  if (lane == 0) *lse_out = lse;
}

}  // namespace

cudaError_t launch_metadata(const int32_t* cache_seqlens, int b, int num_parts, int32_t* metadata,
                            int32_t* num_splits, int32_t* status, cudaStream_t stream) {
  const size_t smem = sizeof(int32_t) * 2 * static_cast<size_t>(b);
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(mla_metadata_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(int32_t) * 2 * kMaxMetadataBatch));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  mla_metadata_kernel<<<1, 256, smem, stream>>>(cache_seqlens, b, num_parts, metadata, num_splits, status);
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
  const int rows = p.s_q * p.h_q;
  dim3 grid(p.b, (rows + 3) / 4);
  mla_combine_kernel<<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
