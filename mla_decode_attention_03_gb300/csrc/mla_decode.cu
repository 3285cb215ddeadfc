// Split-KV MLA decode over a paged latent cache, for sm_103a.
//
// What it computes: for every sequence i, query position j and query head h,
//   out[i,j,h,:] = softmax_t(scale * q[i,j,h,:] . K_t) @ V_t,  lse = ln sum_t e^(...)
// over the visible tokens t of sequence i, where K_t is the 576-dim latent cache
// entry of token t (found through block_table in 64-token pages) and V_t its
// leading 512 dims -- the flash_mla_with_kvcache operation benchmarked by the
// compare_a routine of the PAI FlashMLA tutorial (section 4), over entries of
// stride 576 or the 256-byte aligned 640 of vLLM PR #12676.  The split of the
// KV length across SMs with a log-sum-exp merge is Flash-Decoding's, as the
// Hacker News thread on the FlashMLA release describes it.
//
// Design (one GPU, GB300):
//  * One 2-CTA cluster per scheduler part.  The pair splits the contraction
//    dimension: CTA r owns latent dims [256r, 256r+256) and rope dims
//    [512+32r, 512+32r+32).  Each CTA TMA-loads only its 288 dims of every page
//    (no byte is fetched twice), computes a partial S = Q K^T over them on the
//    tensor cores, and the two partials are swapped through distributed shared
//    memory and summed (a+b == b+a bitwise, so both CTAs hold the same S and take
//    identical softmax decisions).  Each CTA then multiplies P by its own V half
//    (its latent dims are exactly half of V), so O [128 x 512] fp32 -- which
//    would fill all of one SM's tensor memory -- is split 256 columns per SM.
//  * Warp roles per CTA: warp 0 issues TMA, warp 1 issues tcgen05.mma and owns
//    tensor memory, warps 2-5 do the online softmax (one query row per thread)
//    and the epilogue.  All hand-offs are mbarriers; every wait is bounded.
//  * Scores use exp2 with scale*log2(e) folded in; the running max is only
//    moved (and O rescaled in tensor memory) when it grows by more than 8, so
//    rescaling is rare.
#include <cuda_bf16.h>

#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads = 192;
constexpr int kStages = 2;
constexpr int kQChunk = kRowsPerTile * 128;  // 128 rows x 64 bf16 (128B swizzle)
constexpr int kQRope = kRowsPerTile * 64;    // 128 rows x 32 bf16 (64B swizzle)
constexpr int kQBytes = 4 * kQChunk + kQRope;
constexpr int kKChunk = kPage * 128;
constexpr int kKRope = kPage * 64;
constexpr int kKStage = 4 * kKChunk + kKRope;  // 36864 bytes: this CTA's 288 dims of a page
constexpr int kPBuf = kRowsPerTile * 128;      // P: 128 rows x 64 bf16
constexpr int kXRow = 272;                     // exchange row pitch (64 fp32 + 16 B pad)
constexpr int kXBytes = kRowsPerTile * kXRow;

constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;
constexpr int kOffP = kOffK + kStages * kKStage;
constexpr int kOffX = kOffP + 2 * kPBuf;
constexpr int kOffBar = kOffX + kXBytes;

// barrier slots
constexpr int kBarFull = 0;
constexpr int kBarEmpty = kBarFull + kStages;
constexpr int kBarQFull = kBarEmpty + kStages;
constexpr int kBarQEmpty = kBarQFull + 1;
constexpr int kBarSFull = kBarQEmpty + 1;   // 2
constexpr int kBarSEmpty = kBarSFull + 2;   // 2
constexpr int kBarPFull = kBarSEmpty + 2;   // 2
constexpr int kBarPEmpty = kBarPFull + 2;   // 2
constexpr int kBarOFull = kBarPEmpty + 2;
constexpr int kBarXFull = kBarOFull + 1;
constexpr int kBarXEmpty = kBarXFull + 1;
constexpr int kBarDone = kBarXEmpty + 1;
constexpr int kNumBars = kBarDone + 1;

constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemUsed = kOffMisc + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack to align the base to 1024 B

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;     // O half: columns [0, 256)
constexpr uint32_t kTmemS = 256;   // S buffers: [256, 320), [320, 384)

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, false, true);

constexpr float kRescaleThreshold = 8.0f;  // log2 units

// --------------------------------------------------------------- schedule
// One (sequence, page range) piece of a part, and a page-by-page walk over
// all pieces of a part.
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

// ----------------------------------------------------------------- kernel
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
mla_decode_kernel(const __grid_constant__ CUtensorMap q_lat, const __grid_constant__ CUtensorMap q_rope,
                  const __grid_constant__ CUtensorMap k_lat, const __grid_constant__ CUtensorMap k_rope,
                  const DecodeParams P) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw_addr);
  auto bar = [&](int idx) -> uint32_t { return base + kOffBar + 8u * idx; };
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + kOffMisc);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + kOffMisc + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const uint32_t lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int part = blockIdx.x >> 1;
  const int tile = blockIdx.y;
  const int g = blockIdx.z;
  const int32_t* meta = P.metadata + part * kMetaInts;
  const int rows_valid = P.rows_per_tile;

  // ---- setup
  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQEmpty), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarSEmpty + s), 4);
      mbar_init(bar(kBarPFull + s), 4);
      mbar_init(bar(kBarPEmpty + s), 1);
    }
    mbar_init(bar(kBarOFull), 1);
    mbar_init(bar(kBarXFull), 1);
    mbar_init(bar(kBarXEmpty), 4);
    mbar_init(bar(kBarDone), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 2 && rows_valid < kRowsPerTile) {
    // Rows the Q tile does not fill stay zero (their outputs are discarded).
    const int t = tid - 64;
    for (int c = 0; c < 4; ++c)
      for (int off = rows_valid * 128 + t * 16; off < kQChunk; off += 128 * 16)
        *reinterpret_cast<uint4*>(gbase + kOffQ + c * kQChunk + off) = make_uint4(0, 0, 0, 0);
    for (int off = rows_valid * 64 + t * 16; off < kQRope; off += 128 * 16)
      *reinterpret_cast<uint4*>(gbase + kOffQ + 4 * kQChunk + off) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  tc_fence_before_sync();
  cluster_sync();  // barriers of both CTAs are initialised before any remote use
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ================================================= TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&q_lat);
      tma_prefetch_desc(&q_rope);
      tma_prefetch_desc(&k_lat);
      tma_prefetch_desc(&k_rope);
      const uint64_t evict_first = l2_policy_evict_first();
      const int dim_lat = 256 * static_cast<int>(rank);
      const int dim_rope = 512 + 32 * static_cast<int>(rank);
      const uint32_t q_bytes = static_cast<uint32_t>(rows_valid) * 288u * 2u;  // this CTA's 288 dims per row
      PageWalk w;
      w.start(meta, P.cache_seqlens, P.max_blocks);
      int n = 0, qn = 0;
      bool ok = true;
      while (w.valid && ok) {
        if (w.first()) {
          ok = mbar_wait(bar(kBarQEmpty), (qn & 1) ^ 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(kBarQFull), q_bytes);
          const int h0 = g * P.heads_per_kv, j0 = tile * P.q_per_tile;
          for (int c = 0; c < 4; ++c)
            tma_load_4d(base + kOffQ + c * kQChunk, &q_lat, bar(kBarQFull), dim_lat + 64 * c, h0, j0, w.i);
          tma_load_4d(base + kOffQ + 4 * kQChunk, &q_rope, bar(kBarQFull), dim_rope, h0, j0, w.i);
          ++qn;
        }
        int phys = __ldg(P.block_table + static_cast<int64_t>(w.i) * P.max_blocks + w.p);
        if (phys < 0 || phys >= P.num_blocks) {
          raise_status(P.status, kStatusBadBlockId);
          phys = 0;
        }
        const int st = n % kStages;
        ok = mbar_wait(bar(kBarEmpty + st), ((n / kStages) & 1) ^ 1, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(kBarFull + st), kKStage);
        const uint32_t dst = base + kOffK + st * kKStage;
        const int row = phys * kPage;
        for (int c = 0; c < 4; ++c)
          tma_load_3d_hint(dst + c * kKChunk, &k_lat, bar(kBarFull + st), dim_lat + 64 * c, g, row,
                           evict_first);
        tma_load_3d_hint(dst + 4 * kKChunk, &k_rope, bar(kBarFull + st), dim_rope, g, row, evict_first);
        ++n;
        w.advance();
      }
      if (!ok) {
        raise_status(P.status, kStatusTimeout);
        // let the copies already issued land before this CTA can exit
        for (int m = (n > kStages ? n - kStages : 0); m < n; ++m)
          drain_wait(bar(kBarFull + m % kStages), (m / kStages) & 1);
        if (qn > 0) drain_wait(bar(kBarQFull), (qn - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================= MMA issuer
    if (lane == 0) {
      PageWalk wq, wp;
      wq.start(meta, P.cache_seqlens, P.max_blocks);
      wp = wq;
      int nq = 0, np = 0, qn = 0;
      bool ok = true;
      auto issue_qk = [&](const PageWalk& w) -> bool {
        if (w.first()) {
          if (!mbar_wait(bar(kBarQFull), qn & 1, abort_flag)) return false;
          ++qn;
        }
        const int st = nq % kStages;
        if (!mbar_wait(bar(kBarFull + st), (nq / kStages) & 1, abort_flag)) return false;
        const int sb = nq & 1;
        if (!mbar_wait(bar(kBarSEmpty + sb), ((nq >> 1) & 1) ^ 1, abort_flag)) return false;
        tc_fence_after_sync();
        const uint32_t q_s = base + kOffQ;
        const uint32_t k_s = base + kOffK + st * kKStage;
        const uint32_t d = tmem + kTmemS + 64u * sb;
        uint32_t acc = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t a = smem_desc(q_s + c * kQChunk + ks * 32, 16, 1024, kSwizzle128B);
            const uint64_t b = smem_desc(k_s + c * kKChunk + ks * 32, 16, 1024, kSwizzle128B);
            umma_bf16(d, a, b, kIdescQK, acc);
            acc = 1;
          }
        }
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          const uint64_t a = smem_desc(q_s + 4 * kQChunk + ks * 32, 16, 512, kSwizzle64B);
          const uint64_t b = smem_desc(k_s + 4 * kKChunk + ks * 32, 16, 512, kSwizzle64B);
          umma_bf16(d, a, b, kIdescQK, 1);
        }
        umma_commit(bar(kBarSFull + sb));
        if (w.last()) umma_commit(bar(kBarQEmpty));
        ++nq;
        return true;
      };
      auto issue_pv = [&](const PageWalk& w) -> bool {
        const int pb = np & 1;
        if (!mbar_wait(bar(kBarPFull + pb), (np >> 1) & 1, abort_flag)) return false;
        tc_fence_after_sync();
        const int st = np % kStages;
        const uint32_t k_s = base + kOffK + st * kKStage;
        const uint32_t p_s = base + kOffP + pb * kPBuf;
        const uint32_t first = w.first() ? 1u : 0u;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t a = smem_desc(p_s + ks * 32, 16, 1024, kSwizzle128B);
          // V = this CTA's 256 latent dims of the page, read MN-major:
          // 64-dim column blocks 8 KB apart (LBO), 8-token groups 1 KB apart (SBO).
          const uint64_t b = smem_desc(k_s + ks * 2048, kKChunk, 1024, kSwizzle128B);
          umma_bf16(tmem + kTmemO, a, b, kIdescPV, (first && ks == 0) ? 0u : 1u);
        }
        umma_commit(bar(kBarPEmpty + pb));
        umma_commit(bar(kBarEmpty + st));
        umma_commit(bar(kBarOFull));
        ++np;
        return true;
      };
      if (wq.valid) {
        ok = issue_qk(wq);
        wq.advance();
      }
      while (ok && wp.valid) {
        const bool next_same_seg = wq.valid && !wq.first();
        if (next_same_seg) {
          ok = issue_qk(wq);
          wq.advance();
          if (!ok) break;
        }
        ok = issue_pv(wp);
        wp.advance();
        if (!ok) break;
        if (wq.valid && !next_same_seg) {
          ok = issue_qk(wq);
          wq.advance();
        }
      }
      if (!ok) raise_status(P.status, kStatusTimeout);
      umma_commit(bar(kBarDone));
      drain_wait(bar(kBarDone), 0);
    }
    __syncwarp();
  } else {
    // ================================================= softmax + epilogue
    const int quad = warp & 3;
    const int row = 32 * quad + static_cast<int>(lane);
    const uint32_t lane_off = static_cast<uint32_t>(32 * quad) << 16;
    const bool leader = (tid == 64);
    const uint32_t x_row = base + kOffX + row * kXRow;
    const uint32_t peer_x_row = cluster_map(x_row, peer);
    const uint32_t peer_x_full = cluster_map(bar(kBarXFull), peer);
    const uint32_t peer_x_empty = cluster_map(bar(kBarXEmpty), peer);
    uint8_t* const p_gen = gbase + kOffP;

    // row -> (query position, head)
    const int jj = row / P.heads_per_kv;
    const int hh = row - jj * P.heads_per_kv;
    const int j = tile * P.q_per_tile + jj;
    const int h = g * P.heads_per_kv + hh;
    const bool row_live = (row < rows_valid) && (j < P.s_q);
    const int rows_total = P.s_q * P.h_q;
    const int row_in_seq = j * P.h_q + h;

    PageWalk w;
    w.start(meta, P.cache_seqlens, P.max_blocks);
    float m_run = -INFINITY, l_run = 0.f;
    int n = 0;
    bool ok = true;
    int lim = 0;
    while (w.valid && ok) {
      if (w.first()) {
        const int L = __ldg(P.cache_seqlens + w.i);
        lim = P.causal ? L - P.s_q + j + 1 : L;
        lim = min(lim, L);
        m_run = -INFINITY;
        l_run = 0.f;
      }
      const int sb = n & 1;
      if (leader) mbar_arrive_expect_tx(bar(kBarXFull), kRowsPerTile * 256);

      // ---- own partial scores out of tensor memory
      uint32_t s0[32], s1[32];
      ok = mbar_wait(bar(kBarSFull + sb), (n >> 1) & 1, abort_flag);
      if (!ok) break;
      tc_fence_after_sync();
      tmem_ld32(tmem + lane_off + kTmemS + 64u * sb, s0);
      tmem_ld32(tmem + lane_off + kTmemS + 64u * sb + 32, s1);
      tmem_wait_ld2(s0, s1);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarSEmpty + sb));

      // ---- swap partials with the peer CTA
      ok = mbar_wait<true>(bar(kBarXEmpty), (n & 1) ^ 1, abort_flag);
      if (!ok) break;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_async_v4(peer_x_row + 16 * c, s0[4 * c], s0[4 * c + 1], s0[4 * c + 2], s0[4 * c + 3],
                    peer_x_full);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_async_v4(peer_x_row + 128 + 16 * c, s1[4 * c], s1[4 * c + 1], s1[4 * c + 2],
                    s1[4 * c + 3], peer_x_full);
      ok = mbar_wait<true>(bar(kBarXFull), n & 1, abort_flag);
      if (!ok) break;
      float x[64];
      {
        const float4* xr = reinterpret_cast<const float4*>(gbase + kOffX + row * kXRow);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float4 v = xr[c];
          const uint32_t* src = (c < 8) ? &s0[4 * c] : &s1[4 * (c - 8)];
          x[4 * c + 0] = __uint_as_float(src[0]) + v.x;
          x[4 * c + 1] = __uint_as_float(src[1]) + v.y;
          x[4 * c + 2] = __uint_as_float(src[2]) + v.z;
          x[4 * c + 3] = __uint_as_float(src[3]) + v.w;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(peer_x_empty);

      // ---- online softmax for this row and page
      const int t0 = w.p * kPage;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        x[c] = (t0 + c < lim) ? x[c] * P.scale_log2 : -INFINITY;
        mx = fmaxf(mx, x[c]);
      }
      const float m_new = fmaxf(m_run, mx);
      float alpha = 1.f;
      if (m_new > m_run + kRescaleThreshold) {
        alpha = ex2_approx(m_run - m_new);  // 0 when m_run = -inf
        m_run = m_new;
      }
      const float m_sub = (m_run == -INFINITY) ? 0.f : m_run;
      const bool rescale_o = !w.first() && alpha != 1.f;
      if (__any_sync(0xffffffffu, rescale_o)) {
        // O must hold every earlier page before it is scaled.
        ok = mbar_wait(bar(kBarOFull), (n - 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + kTmemO + 32 * c, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tmem + lane_off + kTmemO + 32 * c, o);
        }
        tmem_wait_st();
      }

      // ---- P (bf16) into the swizzled operand buffer
      const int pb = n & 1;
      ok = mbar_wait(bar(kBarPEmpty + pb), ((n >> 1) & 1) ^ 1, abort_flag);
      if (!ok) break;
      float rsum = 0.f;
      uint8_t* prow = p_gen + pb * kPBuf + row * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float e[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          e[u] = ex2_approx(x[8 * c + u] - m_sub);
          rsum += e[u];
        }
        uint4 v;
        v.x = pack_bf16x2(e[0], e[1]);
        v.y = pack_bf16x2(e[2], e[3]);
        v.z = pack_bf16x2(e[4], e[5]);
        v.w = pack_bf16x2(e[6], e[7]);
        *reinterpret_cast<uint4*>(prow + ((c ^ (row & 7)) << 4)) = v;
      }
      l_run = l_run * alpha + rsum;
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull + pb));

      // ---- epilogue at the end of a segment
      if (w.last()) {
        ok = mbar_wait(bar(kBarOFull), n & 1, abort_flag);
        if (!ok) break;
        tc_fence_after_sync();
        const int nsplit = __ldg(P.num_splits + w.i + 1) - __ldg(P.num_splits + w.i);
        const bool direct = (nsplit == 1);
        const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
        const float lse = (l_run > 0.f) ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
        const int64_t slot = static_cast<int64_t>(__ldg(P.num_splits + w.i)) + w.k;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + kTmemO + 32 * c, o);
          tmem_wait_ld(o);
          if (row_live) {
            const int col = 256 * static_cast<int>(rank) + 32 * c;
            if (direct) {
              uint4* dst = reinterpret_cast<uint4*>(
                  static_cast<__nv_bfloat16*>(P.out) +
                  ((static_cast<int64_t>(w.i) * rows_total + row_in_seq) * kDimV + col));
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv_l, __uint_as_float(o[8 * q + 1]) * inv_l);
                v.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv_l, __uint_as_float(o[8 * q + 3]) * inv_l);
                v.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv_l, __uint_as_float(o[8 * q + 5]) * inv_l);
                v.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv_l, __uint_as_float(o[8 * q + 7]) * inv_l);
                dst[q] = v;
              }
            } else {
              float4* dst = reinterpret_cast<float4*>(
                  P.ws_o + ((slot * rows_total + row_in_seq) * kDimV + col));
#pragma unroll
              for (int q = 0; q < 8; ++q)
                dst[q] = make_float4(__uint_as_float(o[4 * q + 0]) * inv_l, __uint_as_float(o[4 * q + 1]) * inv_l,
                                     __uint_as_float(o[4 * q + 2]) * inv_l, __uint_as_float(o[4 * q + 3]) * inv_l);
            }
          }
        }
        if (row_live && rank == 0) {
          if (direct)
            P.lse[(static_cast<int64_t>(w.i) * P.h_q + h) * P.s_q + j] = lse;
          else
            P.ws_lse[slot * rows_total + row_in_seq] = lse;
        }
        tc_fence_before_sync();
      }
      ++n;
      w.advance();
    }
    if (!ok) raise_status(P.status, kStatusTimeout);
  }

  // ---- teardown: everyone is done with tensor memory and with the peer
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();
}

}  // namespace

int decode_smem_bytes() { return kSmemBytes; }

cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& q_lat, const CUtensorMap& q_rope,
                          const CUtensorMap& k_lat, const CUtensorMap& k_rope, int num_parts,
                          int row_tiles, cudaStream_t stream) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  dim3 grid(2 * num_parts, row_tiles, p.h_kv);
  mla_decode_kernel<<<grid, kThreads, kSmemBytes, stream>>>(q_lat, q_rope, k_lat, k_rope, p);
  return cudaGetLastError();
}

cudaError_t decode_max_active_clusters(int* clusters) {
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(clusters, mla_decode_kernel, &cfg);
}

}  // namespace mla
