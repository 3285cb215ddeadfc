// Device helpers shared by the decode kernels: the page walk over one part of
// the split-KV schedule, the status word and the drain wait of the abort path.
#pragma once

#include <cstdint>

#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {

// A page-by-page walk over the (sequence, page range) segments of one part.
struct PageWalk {
  const int32_t* seqlens;
  int max_blocks;
  int i, i_last, pe_last;  // part bounds
  int p, p_begin, p_end;   // current page and its segment's range
  int k;                   // split index of the current segment within its sequence
  bool valid;

  __device__ __forceinline__ static int pages_of(int L, int max_blocks) {
    if (L <= 0) return 0;
    int n = (L + kPage - 1) / kPage;
    return n < max_blocks ? n : max_blocks;
  }
  __device__ __forceinline__ void settle() {
    while (i <= i_last) {
      const int n = pages_of(__ldg(seqlens + i), max_blocks);
      p_end = (i == i_last) ? min(pe_last, n) : n;
      if (p_begin < p_end) {
        p = p_begin;
        valid = true;
        return;
      }
      ++i;
      p_begin = 0;
      k = 0;
    }
    valid = false;
  }
  __device__ __forceinline__ void start(const int32_t* meta, const int32_t* sl, int mb) {
    seqlens = sl;
    max_blocks = mb;
    i = __ldg(meta + 0);
    p_begin = __ldg(meta + 1);
    i_last = __ldg(meta + 2);
    pe_last = __ldg(meta + 3);
    k = __ldg(meta + 4);
    settle();
  }
  __device__ __forceinline__ bool first() const { return p == p_begin; }
  __device__ __forceinline__ bool last() const { return p == p_end - 1; }
  __device__ __forceinline__ void advance() {
    if (++p < p_end) return;
    next_segment();
  }
  __device__ __forceinline__ void next_segment() {
    ++i;
    p_begin = 0;
    k = 0;
    settle();
  }
};

__device__ __forceinline__ void raise_status(int32_t* status, int32_t code) {
  atomicExch(status, code);
}

// Waits that ignore the abort flag: used only to let in-flight asynchronous
// copies land before a CTA that gave up exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitTimeoutCycles) return;
  }
}

}  // namespace mla
