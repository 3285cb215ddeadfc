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
//  * Tensor memory per CTA: O half (256 columns), two S buffers (64 columns
//    each; P overwrites S in place as packed bf16 and feeds PV straight from
//    tensor memory), and the CTA's latent half of Q (128 columns, bf16), so
//    QK reads only K from shared memory.  Shared memory holds 4 K stages, two
//    exchange slots and the rope quarter of Q.
//  * Warp roles per CTA: warp 0 issues TMA, warp 1 issues tcgen05.mma and owns
//    tensor memory, warps 2-5 do the online softmax (one query row per thread)
//    and the epilogue, warps 6-9 stage each sequence's Q into tensor memory.
//    All hand-offs are mbarriers; every wait is bounded.
//  * tcgen05.mma operations of one thread execute in issue order, so QK(n+2)
//    is issued right behind PV(n) into the buffer PV(n) reads P from.
//  * Scores use exp2 with scale*log2(e) folded in; the running max is only
//    moved (and O rescaled in tensor memory) when it grows by more than 8, so
//    rescaling is rare.
#include <cuda_bf16.h>

#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads = 320;
constexpr int kStages = 4;
constexpr int kKChunk = kPage * 128;           // 64 tokens x 64 dims bf16 (128B swizzle)
constexpr int kKRope = kPage * 64;             // 64 tokens x 32 dims bf16 (64B swizzle)
constexpr int kKStage = 4 * kKChunk + kKRope;  // 36864 bytes: this CTA's 288 dims of a page
constexpr int kXSlot = kRowsPerTile * 256;     // exchange: 128 rows x 64 fp32
constexpr int kQRope = kRowsPerTile * 64;      // Q rope quarter: 128 rows x 32 bf16 (64B swizzle)

constexpr int kOffK = 0;
constexpr int kOffX = kOffK + kStages * kKStage;
constexpr int kOffQR = kOffX + 2 * kXSlot;
constexpr int kOffBar = kOffQR + kQRope;

// barrier slots
constexpr int kBarFull = 0;
constexpr int kBarEmpty = kBarFull + kStages;
constexpr int kBarQFull = kBarEmpty + kStages;
constexpr int kBarQEmpty = kBarQFull + 1;
constexpr int kBarSFull = kBarQEmpty + 1;  // 2
constexpr int kBarPFull = kBarSFull + 2;   // 2
constexpr int kBarOFull = kBarPFull + 2;
constexpr int kBarXFull = kBarOFull + 1;   // 2
constexpr int kBarDone = kBarXFull + 2;
constexpr int kNumBars = kBarDone + 1;

constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemUsed = kOffMisc + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack to align the base to 1024 B

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;    // O half: columns [0, 256)
constexpr uint32_t kTmemS = 256;  // S/P buffers: [256, 320), [320, 384)
constexpr uint32_t kTmemQ = 384;  // Q latent half, bf16 pairs: [384, 512)

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, false, true);

constexpr float kRescaleThreshold = 8.0f;  // log2 units

// --------------------------------------------------------------- schedule
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

// Offset of 16-byte chunk c of exchange row r (XOR swizzle: conflict-free for
// both the remote writer and the local reader).
__device__ __forceinline__ uint32_t x_chunk(int r, int c) {
  return static_cast<uint32_t>(r * 256 + ((c ^ (r & 15)) << 4));
}

// ----------------------------------------------------------------- kernel
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
mla_decode_kernel(const __grid_constant__ CUtensorMap q_rope, const __grid_constant__ CUtensorMap k_lat,
                  const __grid_constant__ CUtensorMap k_rope, const DecodeParams P) {
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
    mbar_init(bar(kBarQFull), 1 + 4);  // rope TMA + the 4 Q-staging warps
    mbar_init(bar(kBarQEmpty), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarPFull + s), 4);
      mbar_init(bar(kBarXFull + s), 1);
    }
    mbar_init(bar(kBarOFull), 1);
    mbar_init(bar(kBarDone), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 6 && rows_valid < kRowsPerTile) {
    // Rope rows the Q tile does not fill stay zero (their outputs are discarded).
    const int t = tid - 192;
    for (int off = rows_valid * 64 + t * 16; off < kQRope; off += 128 * 16)
      *reinterpret_cast<uint4*>(gbase + kOffQR + off) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  tc_fence_before_sync();
  cluster_sync();  // barriers of both CTAs are initialised before any remote use
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ================================================= TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&q_rope);
      tma_prefetch_desc(&k_lat);
      tma_prefetch_desc(&k_rope);
      const uint64_t evict_first = l2_policy_evict_first();
      const int dim_lat = 256 * static_cast<int>(rank);
      const int dim_rope = 512 + 32 * static_cast<int>(rank);
      PageWalk w;
      w.start(meta, P.cache_seqlens, P.max_blocks);
      int n = 0, seg = 0;
      bool ok = true;
      while (w.valid && ok) {
        if (w.first()) {
          ok = mbar_wait(bar(kBarQEmpty), (seg & 1) ^ 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(kBarQFull), static_cast<uint32_t>(rows_valid) * 64u);
          tma_load_4d(base + kOffQR, &q_rope, bar(kBarQFull), dim_rope, g * P.heads_per_kv,
                      tile * P.q_per_tile, w.i);
          ++seg;
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
#pragma unroll
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
        if (seg > 0) drain_wait(bar(kBarQFull), (seg - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================= MMA issuer
    if (lane == 0) {
      // Descriptors are built once; per MMA only a constant offset (>> 4) is added.
      const uint64_t d_klat = smem_desc(base + kOffK, 16, 1024, kSwizzle128B);
      const uint64_t d_krope = smem_desc(base + kOffK + 4 * kKChunk, 16, 512, kSwizzle64B);
      const uint64_t d_qrope = smem_desc(base + kOffQR, 16, 512, kSwizzle64B);
      // V = this CTA's 256 latent dims of the page, read MN-major:
      // 64-dim column blocks 8 KB apart (LBO), 8-token groups 1 KB apart (SBO).
      const uint64_t d_v = smem_desc(base + kOffK, kKChunk, 1024, kSwizzle128B);
      PageWalk wq, wp;
      wq.start(meta, P.cache_seqlens, P.max_blocks);
      wp = wq;
      int nq = 0, np = 0, qseg = 0;
      bool ok = true;
      auto issue_qk = [&](const PageWalk& w) -> bool {
        if (w.first()) {
          if (!mbar_wait(bar(kBarQFull), qseg & 1, abort_flag)) return false;
          ++qseg;
        }
        const int st = nq % kStages;
        if (!mbar_wait(bar(kBarFull + st), (nq / kStages) & 1, abort_flag)) return false;
        tc_fence_after_sync();
        const uint32_t d = tmem + kTmemS + 64u * (nq & 1);
        const uint64_t koff = static_cast<uint64_t>((st * kKStage) >> 4);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            umma_bf16_ts(d, tmem + kTmemQ + 32 * c + 8 * ks,
                         d_klat + koff + static_cast<uint64_t>((c * kKChunk + ks * 32) >> 4), kIdescQK,
                         (c | ks) != 0);
          }
        }
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          umma_bf16(d, d_qrope + static_cast<uint64_t>((ks * 32) >> 4),
                    d_krope + koff + static_cast<uint64_t>((ks * 32) >> 4), kIdescQK, 1);
        umma_commit(bar(kBarSFull + (nq & 1)));
        if (w.last()) umma_commit(bar(kBarQEmpty));
        ++nq;
        return true;
      };
      auto issue_pv = [&](const PageWalk& w) -> bool {
        const int pb = np & 1;
        if (!mbar_wait(bar(kBarPFull + pb), (np >> 1) & 1, abort_flag)) return false;
        tc_fence_after_sync();
        const int st = np % kStages;
        const uint64_t voff = static_cast<uint64_t>((st * kKStage) >> 4);
        const uint32_t first = w.first() ? 1u : 0u;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16_ts(tmem + kTmemO, tmem + kTmemS + 64u * pb + 8 * ks,
                       d_v + voff + static_cast<uint64_t>((ks * 2048) >> 4), kIdescPV,
                       (first && ks == 0) ? 0u : 1u);
        umma_commit(bar(kBarEmpty + st));
        umma_commit(bar(kBarOFull));
        ++np;
        return true;
      };
      // QK runs two pages ahead of PV: one S buffer per page in flight.
      for (int a = 0; a < 2 && ok && wq.valid; ++a) {
        ok = issue_qk(wq);
        wq.advance();
      }
      while (ok && wp.valid) {
        ok = issue_pv(wp);
        wp.advance();
        if (ok && wq.valid) {
          ok = issue_qk(wq);  // into the buffer PV just read P from (in-order execution)
          wq.advance();
        }
      }
      if (!ok) raise_status(P.status, kStatusTimeout);
      umma_commit(bar(kBarDone));
      drain_wait(bar(kBarDone), 0);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ================================================= softmax + epilogue
    const int quad = warp & 3;
    const int row = 32 * quad + static_cast<int>(lane);
    const uint32_t lane_off = static_cast<uint32_t>(32 * quad) << 16;
    const bool leader = (tid == 64);
    const uint32_t peer_x = cluster_map(base + kOffX, peer);
    const uint32_t peer_x_full0 = cluster_map(bar(kBarXFull), peer);
    const uint32_t peer_x_full1 = cluster_map(bar(kBarXFull + 1), peer);

    // row -> (query position, head)
    const int jj = row / P.heads_per_kv;
    const int hh = row - jj * P.heads_per_kv;
    const int j = tile * P.q_per_tile + jj;
    const int h = g * P.heads_per_kv + hh;
    const bool row_live = (row < rows_valid) && (j < P.s_q);
    const int rows_total = P.s_q * P.h_q;
    const int row_in_seq = j * P.h_q + h;
    const float c_log2 = P.scale_log2;

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
      const uint32_t par = (n >> 1) & 1;
      if (leader) mbar_arrive_expect_tx(bar(kBarXFull + sb), kXSlot);

      // ---- own partial scores out of tensor memory
      uint32_t s0[32], s1[32];
      ok = mbar_wait(bar(kBarSFull + sb), par, abort_flag);
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t t_s = tmem + lane_off + kTmemS + 64u * sb;
      tmem_ld32(t_s, s0);
      tmem_ld32(t_s + 32, s1);
      tmem_wait_ld2(s0, s1);

      // ---- send them to the peer CTA, take the peer's
      {
        const uint32_t dst = peer_x + sb * kXSlot;
        const uint32_t xb = sb ? peer_x_full1 : peer_x_full0;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_async_v4(dst + x_chunk(row, c), s0[4 * c], s0[4 * c + 1], s0[4 * c + 2], s0[4 * c + 3], xb);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_async_v4(dst + x_chunk(row, 8 + c), s1[4 * c], s1[4 * c + 1], s1[4 * c + 2], s1[4 * c + 3], xb);
      }
      ok = mbar_wait(bar(kBarXFull + sb), par, abort_flag);
      if (!ok) break;
      float x[64];
      {
        const uint8_t* xr = gbase + kOffX + sb * kXSlot;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float4 v = *reinterpret_cast<const float4*>(xr + x_chunk(row, c));
          const uint32_t* src = (c < 8) ? &s0[4 * c] : &s1[4 * (c - 8)];
          x[4 * c + 0] = (__uint_as_float(src[0]) + v.x) * c_log2;
          x[4 * c + 1] = (__uint_as_float(src[1]) + v.y) * c_log2;
          x[4 * c + 2] = (__uint_as_float(src[2]) + v.z) * c_log2;
          x[4 * c + 3] = (__uint_as_float(src[3]) + v.w) * c_log2;
        }
      }

      // ---- online softmax for this row and page
      const int t0 = w.p * kPage;
      if (t0 + kPage > lim) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (t0 + c >= lim) x[c] = -INFINITY;
      }
      float mx8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx8[u] = x[u];
#pragma unroll
      for (int c = 8; c < 64; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], x[c]);
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
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
      }

      // ---- P (bf16 pairs) over S in tensor memory
      uint32_t pk[32];
      float sum8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) sum8[u] = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float e0 = ex2_approx(x[2 * c] - m_sub);
        const float e1 = ex2_approx(x[2 * c + 1] - m_sub);
        sum8[c & 7] += e0 + e1;
        pk[c] = pack_bf16x2(e0, e1);
      }
      tmem_st32(t_s, pk);
      tmem_wait_st();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull + sb));
      const float rsum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      l_run = l_run * alpha + rsum;

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
  } else {
    // ================================================= Q staging into tensor memory
    const int quad = warp & 3;
    const int row = 32 * quad + static_cast<int>(lane);
    const uint32_t lane_off = static_cast<uint32_t>(32 * quad) << 16;
    const int jj = row / P.heads_per_kv;
    const int hh = row - jj * P.heads_per_kv;
    const int j = tile * P.q_per_tile + jj;
    const int h = g * P.heads_per_kv + hh;
    const bool row_live = (row < rows_valid) && (j < P.s_q);
    const __nv_bfloat16* qbase = static_cast<const __nv_bfloat16*>(P.q);

    PageWalk w;
    w.start(meta, P.cache_seqlens, P.max_blocks);
    int seg = 0;
    bool ok = true;
    while (w.valid && ok) {
      // this CTA's 256 latent dims of the row, as 128 bf16 pairs
      uint32_t qr[128];
      if (row_live) {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(
            qbase + ((static_cast<int64_t>(w.i) * P.s_q + j) * P.h_q + h) * kDimQK + 256 * rank);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const uint4 v = ld_global_nc_v4(src + 16 * k);
          qr[4 * k + 0] = v.x;
          qr[4 * k + 1] = v.y;
          qr[4 * k + 2] = v.z;
          qr[4 * k + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < 128; ++k) qr[k] = 0u;
      }
      ok = mbar_wait(bar(kBarQEmpty), (seg & 1) ^ 1, abort_flag);
      if (!ok) break;
      tc_fence_after_sync();
#pragma unroll
      for (int k = 0; k < 4; ++k)
        tmem_st32(tmem + lane_off + kTmemQ + 32 * k, *reinterpret_cast<const uint32_t(*)[32]>(qr + 32 * k));
      tmem_wait_st();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarQFull));
      ++seg;
      w.next_segment();
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

cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& q_rope, const CUtensorMap& k_lat,
                          const CUtensorMap& k_rope, int num_parts, int row_tiles, cudaStream_t stream) {
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
  mla_decode_kernel<<<grid, kThreads, kSmemBytes, stream>>>(q_rope, k_lat, k_rope, p);
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
