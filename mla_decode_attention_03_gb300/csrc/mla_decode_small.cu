// Split-KV MLA decode for tiles of at most 16 query rows (heads per KV head x
// query positions <= 16, as in the DeepSeek-V2-Lite runs of the PAI tutorial,
// section 2: 16 heads, block 64), for sm_103a.
//
// Same operation and the same split-KV schedule, workspace and combine as the
// 128-row kernel (mla_decode.cu).  With 16 rows the 2-CTA cluster of that
// kernel spends a whole 128-row tile (tensor-core instructions of M >= 64, a
// score exchange, eight softmax warps) on an eighth of the work.  Here one CTA
// per part holds everything itself, and the work per page is small enough for
// warp-level tensor-core instructions (m16n8k16, bf16 in, fp32 accumulate),
// operands from shared memory through ldmatrix:
//  * the producer warp loads a segment's Q (16 rows x 576 dims, two buffers)
//    and then its pages, all 576 dims of a page into one of two stages
//    (73,728 B each), each with one TMA copy through a view of the cache whose
//    two innermost dimensions are (64 dims, 9 slices of 64): a stage holds
//    128-byte rows (token, slice) with the 128B swizzle; every page is read
//    once;
//  * four score warps take 16 tokens each: S = Q K^T, the row maxima swapped
//    through shared memory, P = exp(scale (S - m)) as bf16 together with its
//    bf16 rounding error (so P carries ~16 bits), written in the A-fragment
//    order of m16n8k16 with the per-row rescale factor;
//  * four output warps take 128 of the 512 output columns each and add P V
//    into registers, one page behind the score warps (two P buffers);
//  * hand-offs are mbarriers with bounded waits, as in the 128-row kernel.
#include <cuda_bf16.h>

#include "mla_internal.h"
#include "mla_walk.cuh"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

constexpr int kSmScoreWarps = 4;                  // warps 0-3: S, softmax, P
constexpr int kSmOutWarps = 4;                    // warps 4-7: O += P V, epilogue
constexpr int kSmWarps = kSmScoreWarps + kSmOutWarps;
constexpr int kSmThreads = 32 * (kSmWarps + 1);   // + one TMA producer warp (8)
constexpr int kSmRows = 16;
constexpr int kSmStages = 2;
constexpr int kSmBoxes = kDimQK / 64;             // 9 slices of 64 dims (128 B) per token or Q row
constexpr int kSmStage = kPage * kSmBoxes * 128;  // 73728 B: all 576 dims of a page
constexpr int kSmQBuf = kSmRows * kSmBoxes * 128; // 18432 B
// P buffer: hi and lo fragments [chunk of 16 tokens][lane][4 registers] (u32),
// the rescale factor per row, and at a segment's end the score warps' partial
// row sums and the row maxima.
constexpr int kSmPHi = 0;
constexpr int kSmPLo = kSmPHi + 4 * 32 * 16;      // 2048
constexpr int kSmPAlpha = kSmPLo + 4 * 32 * 16;   // 4096: float[16]
constexpr int kSmPL = kSmPAlpha + kSmRows * 4;    // float[4][16]
constexpr int kSmPM = kSmPL + kSmScoreWarps * kSmRows * 4;  // float[16]
constexpr int kSmPBuf = kSmPM + kSmRows * 4;      // 4480 B
constexpr int kSmMxBuf = kSmScoreWarps * kSmRows * 4;       // float[4][16] partial maxima

constexpr int kSmOffK = 0;
constexpr int kSmOffQ = kSmOffK + kSmStages * kSmStage;     // 1024-aligned (swizzle atoms)
constexpr int kSmOffP = kSmOffQ + 2 * kSmQBuf;
constexpr int kSmOffMx = kSmOffP + 2 * kSmPBuf;
constexpr int kSmOffBar = kSmOffMx + 2 * kSmMxBuf;
// barriers, two of each (by stage, segment or page parity), and Stall (never
// completed: the wait-timeout diagnostic waits on it)
constexpr int kSmBarFull = 0;     // TMA bytes of a K stage
constexpr int kSmBarEmpty = 2;    // 8 compute warps are done with a stage
constexpr int kSmBarQFull = 4;    // TMA bytes of a Q buffer
constexpr int kSmBarQEmpty = 6;   // 4 score warps are done with a Q buffer
constexpr int kSmBarMx = 8;       // 4 score warps wrote their partial maxima
constexpr int kSmBarPFull = 10;   // 4 score warps wrote P
constexpr int kSmBarPEmpty = 12;  // 4 output warps read P
constexpr int kSmBarStall = 14;
constexpr int kSmNumBars = 15;
constexpr int kSmOffMisc = kSmOffBar + kSmNumBars * 8;
constexpr int kSmSmemBytes = kSmOffMisc + 16 + 1024;  // abort flag; slack to align the base to 1024 B
static_assert(kSmOffQ % 1024 == 0 && kSmQBuf % 1024 == 0 && kSmStage % 1024 == 0,
              "TMA destinations must sit on 128B-swizzle atoms");
static_assert(kSmOffP % 16 == 0 && kSmPBuf % 16 == 0 && kSmOffBar % 8 == 0, "alignment");
static_assert(kSmSmemBytes <= 232448, "shared memory per CTA");

// Address of 16-byte chunk `chunk` (0..7) of 128-byte row `row` of a region
// that TMA filled with the 128B swizzle from a 1024-byte aligned base (the
// chunk index is XORed with the row index mod 8).  Rows are (token, slice)
// or (Q row, slice) pairs: row = 9 * token + slice.
__device__ __forceinline__ uint32_t sw128(uint32_t base, int row, int chunk) {
  return base + static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const void* map, uint32_t bar, int c0, int c1,
                                                 int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const void* map, uint32_t bar, int c0, int c1, int c2,
                                            int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A B: m16n8k16, A 16x16 bf16 (row), B 16x8 bf16 (col), D fp32.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Lanes that wait on one barrier and give up together: a timed-out wait of
// any lane ends the warp's loop.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
}

__global__ void __launch_bounds__(kSmThreads, 1)
mla_decode_small_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                        const DecodeParams P) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw_addr);
  auto bar = [&](int idx) -> uint32_t { return base + kSmOffBar + 8u * idx; };
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + kSmOffMisc);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int part = blockIdx.x;
  const int g = blockIdx.y;  // KV head
  const int32_t* meta = P.metadata + part * kMetaInts;
  const int hpk = P.heads_per_kv;
  // rows r = jj * hpk + hh of the tile: query position jj, head g * hpk + hh
  const int rows_live = min(kSmRows, P.s_q * hpk);

  // Rows past the live ones are never loaded: zero them once in both Q
  // buffers (the TMA writes only live rows), before any copy can start.
  for (int idx = tid; idx < 2 * kSmQBuf / 16; idx += kSmThreads)
    reinterpret_cast<uint4*>(gbase + kSmOffQ)[idx] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kSmBarFull + s), 1);
      mbar_init(bar(kSmBarEmpty + s), kSmWarps);
      mbar_init(bar(kSmBarQFull + s), 1);
      mbar_init(bar(kSmBarQEmpty + s), kSmScoreWarps);
      mbar_init(bar(kSmBarMx + s), kSmScoreWarps);
      mbar_init(bar(kSmBarPFull + s), kSmScoreWarps);
      mbar_init(bar(kSmBarPEmpty + s), kSmOutWarps);
    }
    mbar_init(bar(kSmBarStall), 1);
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_wait();  // the scheduler's output (and q) are complete from here on
  grid_launch_dependents();

  if (warp == kSmWarps) {
    // ================================================= TMA producer
    if (lane == 0) {
      bool ok = true;
      // Diagnostic: a wait that nothing completes, before any copy is issued
      // (the compute warps then give up on their first wait).
      if (P.stall_test) ok = mbar_wait(bar(kSmBarStall), 0, abort_flag);
      tma_prefetch_desc(&q_map);
      tma_prefetch_desc(&k_map);
      const uint64_t evict_first = l2_policy_evict_first();
      const uint32_t q_bytes = static_cast<uint32_t>(kSmBoxes * 128 * rows_live);
      // The part's first page id, read alongside the walk's own start (a
      // part never starts in an empty sequence), not after it.
      const int i0 = __ldg(meta + 0), p0 = __ldg(meta + 1);
      int phys0 = -1;
      if (i0 >= 0 && i0 < P.b && p0 >= 0 && p0 < P.max_blocks)
        phys0 = __ldg(P.block_table + static_cast<int64_t>(i0) * P.max_blocks + p0);
      PageWalk w;
      w.start(meta, P.cache_seqlens, P.max_blocks);
      int n = 0, seg = 0;
      while (w.valid && ok) {
        if (w.first()) {
          // this segment's Q into buffer seg & 1, once the score warps are
          // done with the segment that used it two segments ago
          const int qb = seg & 1;
          ok = mbar_wait(bar(kSmBarQEmpty + qb), ((seg >> 1) & 1) ^ 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(kSmBarQFull + qb), q_bytes);
          // rows (Q row, slice) = the box {64 dims, 9 slices, hpk heads, s_q positions}
          tma_load_5d(base + kSmOffQ + qb * kSmQBuf, &q_map, bar(kSmBarQFull + qb), 0, 0, g * hpk, 0, w.i);
          ++seg;
        }
        int phys = (n == 0 && w.i == i0 && w.p == p0)
                       ? phys0
                       : __ldg(P.block_table + static_cast<int64_t>(w.i) * P.max_blocks + w.p);
        if (phys < 0 || phys >= P.num_blocks) {
          raise_status(P.status, kStatusBadBlockId);
          phys = 0;
        }
        const int st = n % kSmStages;
        ok = mbar_wait(bar(kSmBarEmpty + st), ((n / kSmStages) & 1) ^ 1, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(kSmBarFull + st), kSmStage);
        // rows (token, slice) = the box {64 dims, 9 slices, 1 KV head, 64 tokens}
        tma_load_4d_hint(base + kSmOffK + st * kSmStage, &k_map, bar(kSmBarFull + st), 0, 0, g, phys * kPage,
                         evict_first);
        ++n;
        w.advance();
      }
      if (!ok) {
        raise_status(P.status, kStatusTimeout);
        // let the copies already issued land before this CTA can exit
        for (int m = (n > kSmStages ? n - kSmStages : 0); m < n; ++m)
          drain_wait(bar(kSmBarFull + m % kSmStages), (m / kSmStages) & 1);
        for (int m = (seg > 2 ? seg - 2 : 0); m < seg; ++m) drain_wait(bar(kSmBarQFull + (m & 1)), (m >> 1) & 1);
      }
    }
    __syncwarp();
    return;
  }

  // Fragment layout of m16n8k16: lane l holds rows gq = l / 4 and gq + 8, and
  // column pairs 2 * (l % 4) of each 8-column tile.
  const int gq = lane >> 2;
  const int qd = lane & 3;
  const float c_log2 = P.scale_log2;
  PageWalk w;
  w.start(meta, P.cache_seqlens, P.max_blocks);
  int n = 0, seg = 0;
  bool ok = true;

  if (warp < kSmScoreWarps) {
    // ================================================= score warps
    // Warp sw takes tokens 16 sw .. 16 sw + 15 of each page.
    const int sw = warp;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    int lim[2] = {0, 0};
    int row_j[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) row_j[u] = (gq + 8 * u) / hpk;
    uint32_t q_base = base + kSmOffQ;
    int qb = 0;
    float* const mx_all = reinterpret_cast<float*>(gbase + kSmOffMx);

    while (ok && w.valid) {
      if (w.first()) {
        qb = seg & 1;
        ok = warp_wait(bar(kSmBarQFull + qb), (seg >> 1) & 1, abort_flag);
        if (!ok) break;
        ++seg;
        q_base = base + kSmOffQ + qb * kSmQBuf;
        const int L = __ldg(P.cache_seqlens + w.i);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          lim[u] = min(P.causal ? L - P.s_q + row_j[u] + 1 : L, L);
          m_run[u] = -INFINITY;
          l_run[u] = 0.f;
        }
      }
      const int st = n % kSmStages;
      ok = warp_wait(bar(kSmBarFull + st), (n / kSmStages) & 1, abort_flag);
      if (!ok) break;
      const uint32_t kst = base + kSmOffK + st * kSmStage;

      // ---- S = Q K^T for this warp's 16 tokens (two 8-token tiles j) over
      // the 576 dims, per 64-dim slice two pairs of k-steps; one accumulator
      // per tile and k-step parity keeps the dependent chains short
      float acc[2][2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][0][e] = acc[j][1][e] = 0.f;
      {
        const int ar = lane & 15, ac = lane >> 4;
        const int bt = 16 * sw + (lane & 7), bc = lane >> 3;
#pragma unroll
        for (int sl = 0; sl < kSmBoxes; ++sl) {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t a0[4], a1[4];
            ldsm_x4(sw128(q_base, kSmBoxes * ar + sl, 4 * h2 + ac), a0[0], a0[1], a0[2], a0[3]);
            ldsm_x4(sw128(q_base, kSmBoxes * ar + sl, 4 * h2 + 2 + ac), a1[0], a1[1], a1[2], a1[3]);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              uint32_t b0, b1, b2, b3;
              ldsm_x4(sw128(kst, kSmBoxes * (bt + 8 * j) + sl, 4 * h2 + bc), b0, b1, b2, b3);
              mma16816(acc[j][0], a0[0], a0[1], a0[2], a0[3], b0, b1);
              mma16816(acc[j][1], a1[0], a1[1], a1[2], a1[3], b2, b3);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(kSmBarEmpty + st));  // the stage's rope dims and K: read
        if (w.last()) mbar_arrive(bar(kSmBarQEmpty + qb));
      }

      // ---- row maxima over the page: this warp's 16 tokens, then the four warps'
      // sv[u][2 j + e]: row gq + 8 u, token 16 sw + 8 j + 2 qd + e
      float sv[2][4];
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) sv[u][2 * j + e] = acc[j][0][2 * u + e] + acc[j][1][2 * u + e];
      const int tb = w.p * kPage + 16 * sw + 2 * qd;
      float* const mxb = mx_all + (n & 1) * (kSmScoreWarps * kSmRows);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if (w.p * kPage + kPage > lim[u]) {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (tb + 8 * (e >> 1) + (e & 1) >= lim[u]) sv[u][e] = -INFINITY;
        }
        float mx = fmaxf(fmaxf(sv[u][0], sv[u][1]), fmaxf(sv[u][2], sv[u][3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        if (qd == 0) mxb[sw * kSmRows + gq + 8 * u] = mx;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kSmBarMx + (n & 1)));
      ok = warp_wait(bar(kSmBarMx + (n & 1)), (n >> 1) & 1, abort_flag);
      if (!ok) break;
      float alpha[2], neg[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int r = gq + 8 * u;
        const float mx = fmaxf(fmaxf(mxb[r], mxb[kSmRows + r]), fmaxf(mxb[2 * kSmRows + r], mxb[3 * kSmRows + r]));
        const float m_new = fmaxf(m_run[u], mx);
        alpha[u] = (m_new == -INFINITY) ? 1.f : ex2_approx((m_run[u] - m_new) * c_log2);  // 0 from -inf
        m_run[u] = m_new;
        neg[u] = (m_new == -INFINITY) ? 0.f : -m_new * c_log2;
        l_run[u] *= alpha[u];
      }

      // ---- P for this warp's tokens: exactly A-fragment chunk sw of the PV
      // step (register u + 2 j: row gq + 8 u, tokens 16 sw + 8 j + 2 qd + {0, 1}),
      // as bf16 (ph) plus its bf16 rounding error (pl)
      uint32_t ph[4], pl[4];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float p0 = ex2_approx(fmaf(sv[u][2 * j], c_log2, neg[u]));
          const float p1 = ex2_approx(fmaf(sv[u][2 * j + 1], c_log2, neg[u]));
          l_run[u] += p0 + p1;
          const uint32_t hi = pack_bf16x2(p0, p1);
          ph[u + 2 * j] = hi;
          pl[u + 2 * j] = pack_bf16x2(p0 - __uint_as_float(hi << 16), p1 - __uint_as_float(hi & 0xffff0000u));
        }
      }
      const int pb = n & 1;
      ok = warp_wait(bar(kSmBarPEmpty + pb), ((n >> 1) & 1) ^ 1, abort_flag);
      if (!ok) break;
      uint8_t* const pbuf = gbase + kSmOffP + pb * kSmPBuf;
      *reinterpret_cast<uint4*>(pbuf + kSmPHi + (sw * 32 + lane) * 16) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
      *reinterpret_cast<uint4*>(pbuf + kSmPLo + (sw * 32 + lane) * 16) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
      float* const pa = reinterpret_cast<float*>(pbuf + kSmPAlpha);
      float* const pls = reinterpret_cast<float*>(pbuf + kSmPL);
      float* const pm = reinterpret_cast<float*>(pbuf + kSmPM);
      if (sw == 0 && qd == 0) {
        pa[gq] = alpha[0];
        pa[gq + 8] = alpha[1];
      }
      if (w.last()) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          float lt = l_run[u] + __shfl_xor_sync(0xffffffffu, l_run[u], 1);
          lt += __shfl_xor_sync(0xffffffffu, lt, 2);
          if (qd == 0) pls[sw * kSmRows + gq + 8 * u] = lt;
          if (sw == 0 && qd == 0) pm[gq + 8 * u] = m_run[u];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kSmBarPFull + pb));
      ++n;
      w.advance();
    }
  } else {
    // ================================================= output warps
    // Warp ov takes output columns 128 ov .. 128 ov + 127: latent slices 2 ov
    // and 2 ov + 1 of each page, one page behind the score warps.
    const int ov = warp - kSmScoreWarps;
    const int rows_total = P.s_q * P.h_q;
    int row_j[2], row_h[2];
    bool row_ok[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int r = gq + 8 * u;
      row_j[u] = r / hpk;
      row_h[u] = g * hpk + (r - row_j[u] * hpk);
      row_ok[u] = r < rows_live;
    }
    // o[b][j]: rows gq (0, 1) and gq + 8 (2, 3), columns 128 ov + 64 b + 8 j + 2 qd + {0, 1}
    float o[2][8][4];
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int j = 0; j < 8; ++j) o[b][j][0] = o[b][j][1] = o[b][j][2] = o[b][j][3] = 0.f;
    int seg_nsplit = 1;
    int64_t seg_oslot = 0;

    while (ok && w.valid) {
      const int pb = n & 1;
      ok = warp_wait(bar(kSmBarPFull + pb), (n >> 1) & 1, abort_flag);
      if (!ok) break;
      const uint8_t* const pbuf = gbase + kSmOffP + pb * kSmPBuf;
      const float* const pa = reinterpret_cast<const float*>(pbuf + kSmPAlpha);
      const float alpha0 = pa[gq], alpha1 = pa[gq + 8];
      const bool last = w.last();
      float lt[2] = {0.f, 0.f}, mrow[2] = {0.f, 0.f};
      if (last) {
        const float* const pls = reinterpret_cast<const float*>(pbuf + kSmPL);
        const float* const pm = reinterpret_cast<const float*>(pbuf + kSmPM);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int r = gq + 8 * u;
          lt[u] = (pls[r] + pls[kSmRows + r]) + (pls[2 * kSmRows + r] + pls[3 * kSmRows + r]);
          mrow[u] = pm[r];
        }
      }

      if (w.first()) {
        // where this segment's rows go: read now, used at its end
        seg_nsplit = __ldg(P.num_splits + w.i + 1) - __ldg(P.num_splits + w.i);
        seg_oslot = static_cast<int64_t>(__ldg(P.num_splits + w.i)) + w.k;
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
          for (int j = 0; j < 8; ++j) o[b][j][0] = o[b][j][1] = o[b][j][2] = o[b][j][3] = 0.f;
      } else {
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            o[b][j][0] *= alpha0;
            o[b][j][1] *= alpha0;
            o[b][j][2] *= alpha1;
            o[b][j][3] *= alpha1;
          }
      }
      // The stage is complete (the score warps waited for it); this wait only
      // gives the output warps their own acquire of the TMA bytes.
      const int st = n % kSmStages;
      ok = warp_wait(bar(kSmBarFull + st), (n / kSmStages) & 1, abort_flag);
      if (!ok) break;
      const uint32_t kst = base + kSmOffK + st * kSmStage;

      // ---- O += P V over the page's 64 tokens, in chunks kc of 16 (P's A
      // fragments for a chunk: one 16-byte load per lane for hi and for lo)
#pragma unroll
      for (int kc = 0; kc < 4; ++kc) {
        const uint4 ph = *reinterpret_cast<const uint4*>(pbuf + kSmPHi + (kc * 32 + lane) * 16);
        const uint4 pl = *reinterpret_cast<const uint4*>(pbuf + kSmPLo + (kc * 32 + lane) * 16);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
#pragma unroll
          for (int jp = 0; jp < 4; ++jp) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(sw128(kst, kSmBoxes * (16 * kc + (lane & 15)) + 2 * ov + b, 2 * jp + (lane >> 4)), b0, b1,
                      b2, b3);
            mma16816(o[b][2 * jp], ph.x, ph.y, ph.z, ph.w, b0, b1);
            mma16816(o[b][2 * jp + 1], ph.x, ph.y, ph.z, ph.w, b2, b3);
            mma16816(o[b][2 * jp], pl.x, pl.y, pl.z, pl.w, b0, b1);
            mma16816(o[b][2 * jp + 1], pl.x, pl.y, pl.z, pl.w, b2, b3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(kSmBarPEmpty + pb));  // P, its row factors and sums: read
        mbar_arrive(bar(kSmBarEmpty + st));   // this warp is done with the stage
      }

      // ---- epilogue at the end of a segment: normalised rows, bf16 to out when
      // the sequence has one segment, else fp32 to its split slot
      if (last) {
        const int nsplit = seg_nsplit;
        const int64_t oslot = seg_oslot;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (!row_ok[u]) continue;
          const float inv = lt[u] > 0.f ? 1.f / lt[u] : 0.f;
          const float lse = lt[u] > 0.f ? (mrow[u] * c_log2 + log2f(lt[u])) * 0.69314718055994531f : -INFINITY;
          const int row_in_seq = row_j[u] * P.h_q + row_h[u];
          if (nsplit == 1) {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(P.out) +
                                 (static_cast<int64_t>(w.i) * rows_total + row_in_seq) * kDimV + 128 * ov + 2 * qd;
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
              for (int j = 0; j < 8; ++j)
                *reinterpret_cast<uint32_t*>(dst + 64 * b + 8 * j) =
                    pack_bf16x2(o[b][j][2 * u] * inv, o[b][j][2 * u + 1] * inv);
            if (ov == 0 && qd == 0)
              P.lse[(static_cast<int64_t>(w.i) * P.h_q + row_h[u]) * P.s_q + row_j[u]] = lse;
          } else {
            float* dst = static_cast<float*>(P.ws_o) + (oslot * rows_total + row_in_seq) * kDimV + 128 * ov + 2 * qd;
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
              for (int j = 0; j < 8; ++j)
                *reinterpret_cast<float2*>(dst + 64 * b + 8 * j) =
                    make_float2(o[b][j][2 * u] * inv, o[b][j][2 * u + 1] * inv);
            if (ov == 0 && qd == 0) P.ws_lse[oslot * rows_total + row_in_seq] = lse;
          }
        }
      }
      ++n;
      w.advance();
    }
  }
  if (!ok) raise_status(P.status, kStatusTimeout);
}

}  // namespace

int decode_small_smem_bytes() { return kSmSmemBytes; }

cudaError_t launch_decode_small(const DecodeParams& p, const CUtensorMap& q_map, const CUtensorMap& k_map, int num_parts,
                                cudaStream_t stream) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(mla_decode_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_parts, p.h_kv, 1);
  cfg.blockDim = dim3(kSmThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_decode_small_kernel, q_map, k_map, p);
}

cudaError_t decode_small_max_ctas(int* ctas) {
  cudaError_t e = cudaFuncSetAttribute(mla_decode_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmSmemBytes);
  if (e != cudaSuccess) return e;
  int per_sm = 0, dev = 0, sms = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mla_decode_small_kernel, kSmThreads, kSmSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  *ctas = per_sm * sms;
  return cudaSuccess;
}

}  // namespace mla
