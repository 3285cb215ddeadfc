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
#include "sm103_ptx.cuh"

namespace mla {
namespace {

// Balanced cut of the (sequence, page) order into num_parts contiguous parts.
//
// Cost axis: sequence i with n_i > 0 pages occupies [C_i, C_i + n_i + F), where
// C is the exclusive prefix sum of the widths and the first F = kSegmentCost
// units stand for the fixed cost of a segment (Q load, epilogue).  Part q takes
// the cost range [q*per, (q+1)*per), per = max(ceil(total/P), kMinPartCost).
// A cut at cost x falls in sequence i = max{i : C_i <= x}, at page
// max(0, x - C_i - F); cuts inside a sequence's first F units therefore start
// the part at that sequence's first page.  Every quantity below is a closed
// form of C and per, so all parts and sequences are computed in parallel.
//
// Output per part:
//   meta[0] = first sequence, meta[1] = first page in it,
//   meta[2] = last sequence,  meta[3] = end page (exclusive) in the last one,
//   meta[4] = split index of the first segment within its sequence.
// An empty part has meta[0] > meta[2].  num_splits[b+1] is the exclusive
// prefix sum of the number of segments (pieces) of each sequence.
constexpr int kMetaThreads = 512;

__device__ __forceinline__ int64_t width_of(int L) {
  const int64_t n = L > 0 ? (static_cast<int64_t>(L) + kPage - 1) / kPage : 0;
  return n > 0 ? n + kSegmentCost : 0;
}

// The last i in [0, b) with C[i] <= x (C[0] = 0 <= x).
__device__ __forceinline__ int seq_at(const int64_t* C, int b, int64_t x) {
  int l = 0, r = b;
  while (l < r) {
    const int m = (l + r) >> 1;
    if (C[m] <= x) l = m + 1; else r = m;
  }
  return l - 1;
}

// Block-wide exclusive scan of one value per thread; returns the block total in *total.
template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T* warp_buf, T* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  T incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_buf[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    T w = lane < kMetaThreads / 32 ? warp_buf[lane] : T(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const T y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kMetaThreads / 32) warp_buf[lane] = w;  // inclusive per-warp prefix
  }
  __syncthreads();
  const T warp_excl = wid > 0 ? warp_buf[wid - 1] : T(0);
  *total = warp_buf[kMetaThreads / 32 - 1];
  __syncthreads();
  return warp_excl + incl - v;
}

__global__ void __launch_bounds__(kMetaThreads) mla_metadata_kernel(const int32_t* __restrict__ seqlens, int b,
                                                                    int num_parts, int32_t* __restrict__ meta,
                                                                    int32_t* __restrict__ num_splits,
                                                                    int32_t* __restrict__ status) {
  extern __shared__ int64_t C[];  // [b + 1]: cost prefix
  __shared__ int64_t buf64[kMetaThreads / 32];
  __shared__ int32_t buf32[kMetaThreads / 32];
  grid_launch_dependents();  // the decode kernel's CTAs may start their set-up
  const int tid = threadIdx.x;
  const int chunk = (b + kMetaThreads - 1) / kMetaThreads;
  const int lo = min(b, tid * chunk), hi = min(b, lo + chunk);

  int64_t local = 0;
  for (int i = lo; i < hi; ++i) {
    const int L = seqlens[i];
    if (L < 0) atomicExch(status, kStatusBadSeqlen);
    local += width_of(L);
  }
  int64_t total = 0;
  int64_t run = block_exclusive_scan<int64_t>(local, buf64, &total);
  for (int i = lo; i < hi; ++i) {
    C[i] = run;
    run += width_of(seqlens[i]);
  }
  if (tid == 0) C[b] = total;
  __syncthreads();

  int64_t per = (total + num_parts - 1) / num_parts;
  if (per < kMinPartCost) per = kMinPartCost;
  auto pages = [&](int i) -> int { return static_cast<int>(C[i + 1] - C[i] - kSegmentCost); };

  for (int q = tid; q < num_parts; q += kMetaThreads) {
    int32_t* m = meta + q * kMetaInts;
    m[5] = m[6] = m[7] = 0;
    const int64_t x0 = static_cast<int64_t>(q) * per;
    const int64_t x1 = x0 + per;
    if (x0 >= total) {
      m[0] = 1; m[1] = 0; m[2] = 0; m[3] = 0; m[4] = 0;
      continue;
    }
    const int i0 = seq_at(C, b, x0);
    const int64_t o0 = x0 - C[i0] - kSegmentCost;
    const int p0 = o0 > 0 ? static_cast<int>(o0) : 0;
    int i1, pe1;
    bool empty = false;
    if (x1 >= total) {
      i1 = seq_at(C, b, total - 1);
      pe1 = pages(i1);
    } else {
      const int ie = seq_at(C, b, x1);
      const int64_t oe = x1 - C[ie] - kSegmentCost;
      if (oe > 0) {
        i1 = ie;
        pe1 = static_cast<int>(oe);
      } else if (ie == i0 && p0 == 0) {
        empty = true;  // both cuts fall before the first page of the same sequence
        i1 = pe1 = 0;
      } else {
        i1 = seq_at(C, b, C[ie] - 1);  // ends with the previous sequence
        pe1 = pages(i1);
      }
    }
    if (empty) {
      m[0] = 1; m[1] = 0; m[2] = 0; m[3] = 0; m[4] = 0;
      continue;
    }
    m[0] = i0;
    m[1] = p0;
    m[2] = i1;
    m[3] = pe1;
    // cuts inside sequence i0 at or before x0: multiples of per in (C + F, x0]
    const int64_t first = (C[i0] + kSegmentCost) / per;
    m[4] = p0 > 0 ? static_cast<int>(q - first) : 0;
  }

  // pieces per sequence: 1 + the cuts strictly inside its pages
  int32_t local_segs = 0;
  for (int i = lo; i < hi; ++i) {
    const int64_t w = C[i + 1] - C[i];
    if (w > 0) local_segs += 1 + static_cast<int32_t>(max(int64_t(0), (C[i] + w - 1) / per - (C[i] + kSegmentCost) / per));
  }
  int32_t seg_total = 0;
  int32_t srun = block_exclusive_scan<int32_t>(local_segs, buf32, &seg_total);
  for (int i = lo; i < hi; ++i) {
    num_splits[i] = srun;
    const int64_t w = C[i + 1] - C[i];
    if (w > 0) srun += 1 + static_cast<int32_t>(max(int64_t(0), (C[i] + w - 1) / per - (C[i] + kSegmentCost) / per));
  }
  if (tid == 0) num_splits[b] = seg_total;
}

// One warp per (sequence, query row).  Sequences with a single split were
// written directly by the decode kernel; sequences with none (length 0) get
// out = 0 and lse = -inf.
constexpr int kCombineWarps = 4;  // rows per block, one warp each

// The common cut, a row in two pieces: both pieces' lse and values in one
// round of loads, then merged (lane l takes columns [16l, 16l+16)).
__device__ __forceinline__ void combine_two(const CombineParams& P, int rows, int row, int s0, int lane,
                                            __nv_bfloat16* out, float* lse_out) {
  const int64_t r0 = static_cast<int64_t>(s0) * rows + row, r1 = r0 + rows;
  const float4* src0 = reinterpret_cast<const float4*>(static_cast<const float*>(P.ws_o) + r0 * kDimV) + lane * 4;
  const float4* src1 = reinterpret_cast<const float4*>(static_cast<const float*>(P.ws_o) + r1 * kDimV) + lane * 4;
  const float l0 = P.ws_lse[r0], l1 = P.ws_lse[r1];
  float4 a[4], b[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    a[q] = src0[q];
    b[q] = src1[q];
  }
  const float m = fmaxf(l0, l1);
  float lse2 = -INFINITY, w0 = 0.f, w1 = 0.f;
  if (m != -INFINITY) {
    const float e0 = expf(l0 - m), e1 = expf(l1 - m);
    const float inv = 1.f / (e0 + e1);
    w0 = e0 * inv;
    w1 = e1 * inv;
    lse2 = m + logf(e0 + e1);
  }
  uint4* dst = reinterpret_cast<uint4*>(out) + lane * 2;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float4 x0 = a[2 * q], x1 = a[2 * q + 1], y0 = b[2 * q], y1 = b[2 * q + 1];
    __nv_bfloat162 c0 = __floats2bfloat162_rn(w0 * x0.x + w1 * y0.x, w0 * x0.y + w1 * y0.y);
    __nv_bfloat162 c1 = __floats2bfloat162_rn(w0 * x0.z + w1 * y0.z, w0 * x0.w + w1 * y0.w);
    __nv_bfloat162 c2 = __floats2bfloat162_rn(w0 * x1.x + w1 * y1.x, w0 * x1.y + w1 * y1.y);
    __nv_bfloat162 c3 = __floats2bfloat162_rn(w0 * x1.z + w1 * y1.z, w0 * x1.w + w1 * y1.w);
    uint4 v;
    v.x = *reinterpret_cast<uint32_t*>(&c0);
    v.y = *reinterpret_cast<uint32_t*>(&c1);
    v.z = *reinterpret_cast<uint32_t*>(&c2);
    v.w = *reinterpret_cast<uint32_t*>(&c3);
    dst[q] = v;
  }
  if (lane == 0) *lse_out = lse2;
}

__global__ void __launch_bounds__(32 * kCombineWarps) mla_combine_kernel(const CombineParams P) {
  grid_dependency_wait();  // the decode kernel's partials are complete and visible
  const int i = blockIdx.x;
  const int rows = P.s_q * P.h_q;
  const int row = blockIdx.y * kCombineWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int s0 = P.num_splits[i];
  const int ns = P.num_splits[i + 1] - s0;
  if (ns == 1) return;
  const int j = row / P.h_q, h = row - (row / P.h_q) * P.h_q;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(P.out) + (static_cast<int64_t>(i) * rows + row) * kDimV;
  float* lse_out = P.lse + (static_cast<int64_t>(i) * P.h_q + h) * P.s_q + j;

  if (ns == 2) {
    combine_two(P, rows, row, s0, lane, out, lse_out);
    return;
  }

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
      // lane l merges columns [16l, 16l+16): four 16-byte loads of fp32
      const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(P.ws_o) + r * kDimV) + lane * 4;
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

// The same merge when many pieces per sequence are expected (the schedule
// has at least twice as many parts as sequences): four warps per row, each
// taking every fourth piece of the row, so that four chains of loads are in
// flight per row, their sums added through shared memory.  A block still
// covers 4 rows of one sequence.
constexpr int kCombineSplit = 4;  // warps per row

__global__ void __launch_bounds__(32 * kCombineWarps * kCombineSplit, 1) mla_combine_many_kernel(const CombineParams P) {
  __shared__ float4 red[kCombineSplit - 1][kCombineWarps][4][32];  // the other warps' sums, [q][lane] per row
  grid_dependency_wait();  // the decode kernel's partials are complete and visible
  const int i = blockIdx.x;
  const int rows = P.s_q * P.h_q;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rw = warp % kCombineWarps;   // row within the block
  const int part = warp / kCombineWarps;  // which of the row's warps
  const int row = blockIdx.y * kCombineWarps + rw;
  const bool live = row < rows;
  const int s0 = P.num_splits[i];
  const int ns = P.num_splits[i + 1] - s0;  // the same for the whole block
  if (ns == 1) return;
  const int j = row / P.h_q, h = row - (row / P.h_q) * P.h_q;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(P.out) + (static_cast<int64_t>(i) * rows + row) * kDimV;
  float* lse_out = P.lse + (static_cast<int64_t>(i) * P.h_q + h) * P.s_q + j;
  const float* ws_o = static_cast<const float*>(P.ws_o);
  if (ns == 2) {  // the same for the whole block: no barrier below is reached
    if (part == 0 && live) combine_two(P, rows, row, s0, lane, out, lse_out);
    return;
  }

  // every warp of a row forms the row's lse from all pieces' lse, then adds
  // its own pieces' weighted values (no piece: out = 0, lse = -inf)
  float4 acc[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  float lse = -INFINITY;
  if (live && ns > 0) {
    float mx = -INFINITY;
    for (int k = lane; k < ns; k += 32) mx = fmaxf(mx, P.ws_lse[static_cast<int64_t>(s0 + k) * rows + row]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (mx != -INFINITY) {
      float sum = 0.f;
      for (int k = lane; k < ns; k += 32) sum += expf(P.ws_lse[static_cast<int64_t>(s0 + k) * rows + row] - mx);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      lse = mx + logf(sum);
      for (int k = part; k < ns; k += kCombineSplit) {
        const int64_t r = static_cast<int64_t>(s0 + k) * rows + row;
        const float wgt = expf(P.ws_lse[r] - lse);
        // lane l merges columns [16l, 16l+16): four 16-byte loads of fp32
        const float4* src = reinterpret_cast<const float4*>(ws_o + r * kDimV) + lane * 4;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 v = src[q];
          acc[q].x += wgt * v.x;
          acc[q].y += wgt * v.y;
          acc[q].z += wgt * v.z;
          acc[q].w += wgt * v.w;
        }
      }
    }
  }
  if (part > 0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) red[part - 1][rw][q][lane] = acc[q];
  }
  __syncthreads();
  if (part != 0 || !live) return;
#pragma unroll
  for (int o = 0; o < kCombineSplit - 1; ++o) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v = red[o][rw][q][lane];
      acc[q].x += v.x;
      acc[q].y += v.y;
      acc[q].z += v.z;
      acc[q].w += v.w;
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(out) + lane * 2;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    __nv_bfloat162 a = __floats2bfloat162_rn(acc[2 * q].x, acc[2 * q].y);
    __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * q].z, acc[2 * q].w);
    __nv_bfloat162 c = __floats2bfloat162_rn(acc[2 * q + 1].x, acc[2 * q + 1].y);
    __nv_bfloat162 d = __floats2bfloat162_rn(acc[2 * q + 1].z, acc[2 * q + 1].w);
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
  const size_t smem = sizeof(int64_t) * (static_cast<size_t>(b) + 1);
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(mla_metadata_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sizeof(int64_t) * (kMaxMetadataBatch + 1)));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  mla_metadata_kernel<<<1, kMetaThreads, smem, stream>>>(cache_seqlens, b, num_parts, metadata, num_splits, status);
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
  const int rows = p.s_q * p.h_q;
  // Many pieces per sequence (at least twice as many parts as sequences, as
  // with small batches on one CTA per SM): four warps per row.  Otherwise
  // mostly one or two pieces: one warp per row, four rows per block.
  const bool many = p.num_parts >= 2 * p.b;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.b, (rows + kCombineWarps - 1) / kCombineWarps, 1);
  cfg.blockDim = dim3(32 * kCombineWarps * (many ? kCombineSplit : 1), 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return many ? cudaLaunchKernelEx(&cfg, mla_combine_many_kernel, p) : cudaLaunchKernelEx(&cfg, mla_combine_kernel, p);
}

}  // namespace mla
