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
//    (no byte is fetched twice) and computes a partial S = Q K^T over them on the
//    tensor cores.  The partials are swapped through distributed shared memory
//    as int16 with one fp32 scale per (row, 32 tokens) -- half the bytes of fp32,
//    which matters because SM-to-SM bandwidth, not HBM, bounds this exchange.
//    Each CTA adds its own exact fp32 partial to the dequantised peer partial, so
//    the two CTAs see scores that differ by at most one quantisation step
//    (1/32767 of the largest partial of that row and 32 tokens); each CTA runs its own
//    online softmax and normalises its own output half with its own sums.  Each
//    CTA multiplies P by its own V half (its latent dims are exactly half of V),
//    so O [128 x 512] fp32 -- which would fill all of one SM's tensor memory --
//    is split 256 columns per SM.
//  * Tensor memory per CTA: O half (256 columns), two S buffers (64 columns
//    each), one P buffer (32 columns of packed bf16 that feed PV straight from
//    tensor memory) and 192 of the CTA's 256 latent Q dims (96 columns); the
//    other 64 latent Q dims and the CTA's 32 rope dims sit in shared memory.
//  * Warp roles per CTA (four warpgroups, registers moved by setmaxnreg):
//    warps 0-3 stage each sequence's Q and, per page, read the CTA's partial S
//    out of tensor memory, quantise it and send it to the peer; warp 4 issues
//    TMA; warp 5 issues PV and owns tensor memory; warps 6 and 7 issue QK for
//    even and odd pages; warps 8-15 run the online softmax
//    and the epilogue, each over 16 full rows (half a tensor-memory lane
//    quadrant) and all 64 tokens of a page, so a row's max and sum need one
//    warp shuffle and no other warp.
//  * Page n flows in order: QK(n) -> the sender warps quantise and send the
//    partial while the softmax warps read theirs -> the peer's partial lands ->
//    softmax -> P -> PV(n).  QK runs up to two pages ahead of the softmax (two
//    S buffers, each handed back as soon as the softmax has read it); five K
//    stages hide most of the HBM latency under load (with four the bench
//    workload ran 5% slower; a sixth does not fit shared memory).  Holding
//    QK back until PV(n-3) had been issued, or prefetching S a page early, was
//    measured slower and dropped.
//  * P is rounded to bf16 for the tensor cores.  On pages where one weight
//    exceeds a third of its row's running sum, a second PV pass adds
//    P_lo V (P_lo = the bf16 rounding error of P, itself in bf16), so cancelling
//    value rows under a few dominant keys stay within the tolerance.
//  * Exchange slots are returned to the sender by an explicit credit: each
//    softmax warp that has read its part of a slot fences (CTA scope) and
//    counts; the warp that completes the count of 8 sends one relaxed remote
//    arrive to the peer's sender barrier, so no slot is overwritten before it
//    is read.  (A release-ordered remote arrive from every warp cost 70 us per
//    decode; an unordered relaxed one from every warp raced.)  All other
//    hand-offs are mbarriers; every wait is bounded.
//  * Scores use exp2 with scale*log2(e) folded in; the running max is only
//    moved (and O rescaled in tensor memory) when it grows by more than 8, so
//    rescaling is rare.
#include <cuda_bf16.h>

#include "mla_internal.h"
#include "mla_walk.cuh"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads = 512;
constexpr int kFirstSoftmaxWarp = 8;
// Registers (setmaxnreg): launched at 128 per thread; the issuing warpgroup
// (warps 4-7) drops to 48 and the staging/sending warpgroup (warps 0-3) to 120,
// the two softmax warpgroups take the rest: 128*48 + 128*120 + 256*168 <= 512*128.
constexpr uint32_t kRegsIssue = 48;
constexpr uint32_t kRegsStage = 120;
constexpr uint32_t kRegsSoftmax = 168;
// setmaxnreg.inc waits until the registers it asks for are free: the three
// shares must fit in what the block was launched with (128 per thread).
static_assert(128 * kRegsIssue + 128 * kRegsStage + 256 * kRegsSoftmax <= kThreads * 128u,
              "register split exceeds the launch allocation");
// A K stage is held from its TMA issue (microseconds of HBM latency under
// load) until the PV of its page has read V, so the number of stages bounds the
// pages in flight; five stages and a single exchange slot fill the 227 KB.
constexpr int kStages = 5;
constexpr int kKChunk = kPage * 128;           // 64 tokens x 64 dims bf16 (128B swizzle)
constexpr int kKRope = kPage * 64;             // 64 tokens x 32 dims bf16 (64B swizzle)
constexpr int kKStage = 4 * kKChunk + kKRope;  // 36864 bytes: this CTA's 288 dims of a page
constexpr int kXSlots = 1;     // receive slots (peer partials)
constexpr int kXData = kRowsPerTile * 128;     // 128 rows x 64 int16 (two 32-token halves)
constexpr int kXSlot = kXData + 2 * kRowsPerTile * 4;  // + one fp32 scale per (row, half)
constexpr int kXRowBytes = kXSlot / kRowsPerTile;      // one row's share: 136 bytes
constexpr int kQRope = kRowsPerTile * 64;      // the CTA's 32 Q rope dims: 128 rows x 32 bf16 (64B swizzle)
constexpr int kQLat = kRowsPerTile * 128;      // Q latent dims [192, 256) of the CTA: 128 rows x 64 bf16

constexpr int kOffK = 0;
constexpr int kOffX = kOffK + kStages * kKStage;
constexpr int kOffQL = kOffX + kXSlots * kXSlot;  // 1024-aligned (128B swizzle atom)
constexpr int kOffQR = kOffQL + kQLat;
constexpr int kOffBar = kOffQR + kQRope;

// barrier slots
constexpr int kBarFull = 0;
constexpr int kBarEmpty = kBarFull + kStages;
constexpr int kBarQFull = kBarEmpty + kStages;
constexpr int kBarQEmpty = kBarQFull + 1;
constexpr int kBarSFull = kBarQEmpty + 1;   // 2
constexpr int kBarSFree = kBarSFull + 2;    // 2
constexpr int kBarPFull = kBarSFree + 2;
constexpr int kBarOFull = kBarPFull + 1;
constexpr int kBarXFull = kBarOFull + 1;    // kXSlots
constexpr int kBarXEmpty = kBarXFull + kXSlots;  // kXSlots: the peer has read the slot
constexpr int kBarDone = kBarXEmpty + kXSlots;
constexpr int kBarStall = kBarDone + 1;  // never completed: the wait-timeout diagnostic waits on it
constexpr int kNumBars = kBarStall + 1;

constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kOffLoFlag = kOffMisc + 16 + 4 * kXSlots;  // two words: page (by parity) + 1 when its low part runs
constexpr int kSmemUsed = kOffLoFlag + 8;  // tmem slot, abort flag, pad, slot-read counters, low-part flags
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack to align the base to 1024 B
static_assert(kOffQL % 1024 == 0, "Q latent tile must sit on a 128B-swizzle atom");
static_assert(kOffQR % 512 == 0, "Q rope tile must sit on a 64B-swizzle atom");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;    // O half: columns [0, 256)
constexpr uint32_t kTmemS = 256;  // S buffers: [256, 320), [320, 384)
constexpr uint32_t kTmemP = 384;  // P, bf16 pairs: [384, 416)
constexpr uint32_t kTmemQ = 416;  // Q latent dims [0, 192) of the CTA, bf16 pairs: [416, 512)

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, false, true);

constexpr float kRescaleThreshold = 8.0f;  // log2 units
// A page gets a second PV pass with the bf16 rounding error of P (P - bf16(P),
// itself in bf16) when one of its weights exceeds a third of its row's running
// sum, this page included: 3 * e > l.  Such weights carry enough of the output
// that the 2^-9 relative rounding of P alone could move an output element by
// more than the tolerance when value rows cancel.  (Many weights of similar
// size, as on the first page of a segment, round independently and need no
// second pass.)
constexpr float kLoRatio = 3.0f;
constexpr float kQuantMax = 32767.0f;
// q in [-32767, 32767] travels as the low 16 bits of the fp32 value
// 1.5*2^23 + 32768 + q, whose unit in the last place is 1: one FMA rounds and
// encodes, one byte permute and one subtraction decode.
constexpr float kQuantBase = 12615680.0f;  // 1.5 * 2^23 + 32768
constexpr uint32_t kQuantHi = 0x4B400000u;  // upper half of the bit pattern of 1.5 * 2^23

// Exchange slot layout: softmax thread (warp w, lane l) of one CTA sends its
// 64 bytes of int16 scores to the thread (w, l) of the peer, which is the only
// reader.  Chunk k of that thread sits at ((w*4 + k)*32 + l)*16, so each warp
// instruction writes (and later reads) 512 contiguous bytes; its fp32 scale at
// kXData + (w*32 + l)*4.
__device__ __forceinline__ uint32_t x_chunk(int sw, int lane, int k) {
  return static_cast<uint32_t>(((sw * 4 + k) * 32 + lane) * 16);
}

__device__ __forceinline__ uint32_t x_scale(int sw, int lane) {
  return static_cast<uint32_t>(kXData + (sw * 32 + lane) * 4);
}

// O <- alpha * O for this warp's 16 rows of the CTA's O half (columns
// [0, 256) of tensor memory from `t_o`), in eight 32-column steps.
__device__ __noinline__ void rescale_o_half(uint32_t t_o, float alpha) {
#pragma unroll 1
  for (int c = 0; c < 8; ++c) {
    uint32_t o[16];
    tmem_ld16x2(t_o + 32u * c, o);
    tmem_wait_ld16(o);
#pragma unroll
    for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
    tmem_st16x2(t_o + 32u * c, o);
  }
}

// In-register transpose of 16-byte blocks within each group of G lanes (G = 4
// or 8): lane G*a + m enters with the G blocks b[4j .. 4j+3] of its own output
// line and leaves with block m of the lines of lanes G*a + [0, G), in lane
// order.  log2(G) butterfly steps; each swaps the half of the blocks whose
// index differs from the lane in one bit with the partner lane across it.
template <int G>
__device__ __forceinline__ void transpose_blocks(uint32_t (&b)[4 * G], int lane) {
#pragma unroll
  for (int bit = G / 2; bit >= 1; bit >>= 1) {
    const bool up = (lane & bit) != 0;
#pragma unroll
    for (int j0 = 0; j0 < G; ++j0) {
      if (j0 & bit) continue;
      const int j1 = j0 | bit;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, up ? b[4 * j0 + e] : b[4 * j1 + e], bit);
        if (up)
          b[4 * j0 + e] = recv;
        else
          b[4 * j1 + e] = recv;
      }
    }
  }
}

// Writes this warp's 16 rows of the CTA's O half (tensor memory from `t_o`),
// scaled by each row's 1/l, to global memory: bf16 into `out_b` or fp32 into
// `out_f` (row r of the segment at element r * kDimV, this CTA's half at
// `col0`).  Lane l holds row l & 15, columns 32 * (l >> 4) + [0, 32) of a
// 64-column chunk; a transpose within groups of lanes lets every store
// instruction write four whole 128-byte lines instead of touching 32 lines
// with 16 bytes each.  Rows whose bit in `live` is clear are not written.
__device__ __noinline__ void write_o_rows(uint32_t t_o, float inv_l, __nv_bfloat16* out_b, float* out_f, int col0,
                                          int row_in_seq, uint32_t live) {
  const int lane = static_cast<int>(lane_id());
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t o[32];
    tmem_ld16x2_32(t_o + 64u * c, o);
    tmem_wait_ld(o);
    if (out_b != nullptr) {
      // a line is one row's 64 columns (two lanes' 64 bytes): groups of four
      // lanes hold four rows of one half; lanes 4a+m and 4(a+4)+m write the
      // two halves of row 4(a & 3) + k
      uint32_t b[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        b[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
      transpose_blocks<4>(b, lane);
      const int a = lane >> 2, m = lane & 3;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int rs = 4 * (a & 3) + k;
        const int64_t r = __shfl_sync(0xffffffffu, row_in_seq, rs);
        if ((live >> rs) & 1u)
          *reinterpret_cast<uint4*>(out_b + r * kDimV + col0 + 64 * c + 32 * (a >> 2) + 8 * m) =
              make_uint4(b[4 * k], b[4 * k + 1], b[4 * k + 2], b[4 * k + 3]);
      }
    } else {
      // a line is one row's 32 columns of one half (one lane's 128 bytes):
      // groups of eight lanes hold eight rows of one half
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * inv_l);
      transpose_blocks<8>(o, lane);
      const int a = lane >> 3, m = lane & 7;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int rs = 8 * (a & 1) + k;
        const int64_t r = __shfl_sync(0xffffffffu, row_in_seq, rs);
        if ((live >> rs) & 1u)
          *reinterpret_cast<uint4*>(out_f + r * kDimV + col0 + 64 * c + 32 * (a >> 1) + 4 * m) =
              make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
      }
    }
  }
}

// The low-part pass of page `page`, run by every softmax warp once all of them
// have handed that page's bf16 P over (the PFull phase `groups - 1`): if any
// warp asked for it (the flag holds page + 1), wait until the bf16 part's PV
// has read the P buffer, store this warp's low part (zero where it did not
// ask) and hand it over as one more PV group.  Returns false on abort.
__device__ __forceinline__ bool lo_pass(uint32_t pfull, uint32_t ofull, volatile int* lo_flag, int page, int& groups,
                                        uint32_t t_p, const uint32_t (&lo)[16], volatile int* abort_flag) {
  if (!mbar_wait(pfull, (groups - 1) & 1, abort_flag)) return false;  // every warp's request is in
  if (lo_flag[page & 1] != page + 1) return true;
  if (!mbar_wait(ofull, (groups - 1) & 1, abort_flag)) return false;
  tc_fence_after_sync();
  tmem_st16x2(t_p, lo);
  tmem_wait_st();
  tc_fence_before_sync();
  __syncwarp();
  if (lane_id() == 0) mbar_arrive(pfull);
  ++groups;
  return mbar_wait(ofull, (groups - 1) & 1, abort_flag);  // the low part's PV is complete
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
  uint32_t* const xread_cnt = reinterpret_cast<uint32_t*>(gbase + kOffMisc + 16);  // [kXSlots]
  volatile int* const lo_flag = reinterpret_cast<volatile int*>(gbase + kOffLoFlag);  // [2]

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
  // Rows of this tile that belong to a query position: a prefix of the tile.
  // Only they are exchanged (a tile of 16 heads sends an eighth of the bytes).
  const int rows_live = min(rows_valid, (P.s_q - tile * P.q_per_tile) * P.heads_per_kv);

  // ---- setup
  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kXSlots; ++s) xread_cnt[s] = 0;
    lo_flag[0] = 0;
    lo_flag[1] = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    mbar_init(bar(kBarQFull), 1 + 4);  // rope TMA + the 4 Q-staging warps
    mbar_init(bar(kBarQEmpty), 2);  // both QK issuers
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarSFree + s), 8 + 4);  // softmax warps + sender warps
    }
    mbar_init(bar(kBarPFull), 8);
    mbar_init(bar(kBarOFull), 1);
    for (int s = 0; s < kXSlots; ++s) {
      mbar_init(bar(kBarXFull + s), 1);
      mbar_init(bar(kBarXEmpty + s), 1);
    }
    mbar_init(bar(kBarDone), 3);    // the three MMA-issuing threads
    mbar_init(bar(kBarStall), 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp < 4 && rows_valid < kRowsPerTile) {
    // Rope rows the Q tile does not fill stay zero (their outputs are discarded).
    const int t = tid;
    for (int off = rows_valid * 64 + t * 16; off < kQRope; off += 128 * 16)
      *reinterpret_cast<uint4*>(gbase + kOffQR + off) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  tc_fence_before_sync();
  cluster_sync();  // barriers of both CTAs are initialised before any remote use
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // Everything above overlaps the previous kernel (the scheduler); nothing it
  // wrote is read before this point.
  grid_dependency_wait();
  grid_launch_dependents();

  // Warpgroups: 0-3 stage Q and send the exchange, 4-7 issue TMA and MMA, 8-15
  // run the softmax.  Each warpgroup sets its register count as a whole.
  if (warp >= 4 && warp < 8) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsIssue));
  if (warp == 4) {
    // ================================================= TMA producer
    if (lane == 0) {
      bool ok = true;
      if (P.stall_test) {
        // Diagnostic: a wait that nothing completes, before any copy is
        // issued.  The bounded wait gives up, raises the abort flag and every
        // other warp role leaves its own wait; the call reports a timeout.
        ok = mbar_wait(bar(kBarStall), 0, abort_flag);
      }
      tma_prefetch_desc(&k_lat);
      tma_prefetch_desc(&k_rope);
      const uint64_t evict_first = l2_policy_evict_first();
      const int dim_lat = 256 * static_cast<int>(rank);
      const int dim_rope = 512 + 32 * static_cast<int>(rank);
      PageWalk w;
      w.start(meta, P.cache_seqlens, P.max_blocks);
      // (Prefetching pages into L2 ahead of their TMA loads was measured and
      // dropped: 2, 4 and 8 pages ahead all ran slower than none.)
      // The Q rows of every later segment of this part go to L2 now: a
      // segment's Q is staged only once the previous segment's QKs are done,
      // and read from HBM that staging stalled the pipeline for microseconds.
      if (ok) {
        PageWalk ws = w;
        if (ws.valid) ws.next_segment();
        const uint8_t* const qb = static_cast<const uint8_t*>(P.q);
        const uint32_t row_bytes = static_cast<uint32_t>(P.heads_per_kv) * kDimQK * 2u;
        for (; ws.valid; ws.next_segment()) {
          for (int jj = 0; jj < P.q_per_tile; ++jj) {
            const int jq = tile * P.q_per_tile + jj;
            if (jq >= P.s_q) break;
            const uint8_t* src = qb + ((static_cast<int64_t>(ws.i) * P.s_q + jq) * P.h_q +
                                       static_cast<int64_t>(g) * P.heads_per_kv) * (kDimQK * 2);
            for (uint32_t off = 0; off < row_bytes; off += 16384u)
              bulk_prefetch_l2(src + off, min(16384u, row_bytes - off));
          }
        }
      }
      // K pages need no Q: the loads run on across segment boundaries (a
      // segment's Q rope dims are loaded by the Q-staging warps).
      int n = 0;
      while (w.valid && ok) {
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
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ================================================= PV issuer
    // Warp 5 issues PV; QK is issued by warps 6 and 7 (even and odd pages).
    // Splitting the tcgen05.mma issue over three sub-partitions keeps any one of
    // them from starving the two softmax warps it hosts (one thread issues at
    // most one MMA per ~52 cycles, so the 18 N=64 MMAs of a page's QK take about
    // 950 cycles to issue).
    if (lane == 0) {
      // V = this CTA's 256 latent dims of the page, read MN-major:
      // 64-dim column blocks 8 KB apart (LBO), 8-token groups 1 KB apart (SBO).
      const uint64_t d_v = smem_desc(base + kOffK, kKChunk, 1024, kSwizzle128B);
      PageWalk wp;
      wp.start(meta, P.cache_seqlens, P.max_blocks);
      int np = 0, kp = 0;  // pages, P hand-offs
      bool ok = true;
      while (wp.valid) {
        ok = mbar_wait(bar(kBarPFull), kp & 1, abort_flag);
        if (!ok) break;
        ++kp;
        tc_fence_after_sync();
        const int st = np % kStages;
        const uint64_t voff = static_cast<uint64_t>((st * kKStage) >> 4);
        const uint32_t first = wp.first() ? 1u : 0u;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16_ts(tmem + kTmemO, tmem + kTmemP + 8 * ks,
                       d_v + voff + static_cast<uint64_t>((ks * 2048) >> 4), kIdescPV,
                       (first && ks == 0) ? 0u : 1u);
        // the softmax warps asked for the low part of this page's P (visible:
        // written before their arrivals on the barrier just waited on)
        const bool lo = (lo_flag[np & 1] == np + 1);
        if (!lo) umma_commit(bar(kBarEmpty + st));
        umma_commit(bar(kBarOFull));
        if (lo) {
          ok = mbar_wait(bar(kBarPFull), kp & 1, abort_flag);
          if (!ok) break;
          ++kp;
          tc_fence_after_sync();
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_bf16_ts(tmem + kTmemO, tmem + kTmemP + 8 * ks,
                         d_v + voff + static_cast<uint64_t>((ks * 2048) >> 4), kIdescPV, 1u);
          umma_commit(bar(kBarEmpty + st));
          umma_commit(bar(kBarOFull));
        }
        ++np;
        wp.advance();
      }
      if (!ok) raise_status(P.status, kStatusTimeout);
      umma_commit(bar(kBarDone));
      drain_wait(bar(kBarDone), 0);
    }
    __syncwarp();
  } else {
    // ================================================= QK issuers
    // Warp 6 takes the even pages (S buffer 0, K stages 0 and 2), warp 7 the
    // odd ones.  QK(k) needs S buffer k&1 back from the softmax (it has read
    // S(k-2)), the page's K stage and its segment's Q.
    if (lane == 0) {
      const int parity = warp - 6;
      const uint64_t d_klat = smem_desc(base + kOffK, 16, 1024, kSwizzle128B);
      const uint64_t d_krope = smem_desc(base + kOffK + 4 * kKChunk, 16, 512, kSwizzle64B);
      const uint64_t d_qlat = smem_desc(base + kOffQL, 16, 1024, kSwizzle128B);
      const uint64_t d_qrope = smem_desc(base + kOffQR, 16, 512, kSwizzle64B);
      const uint32_t d = tmem + kTmemS + 64u * static_cast<uint32_t>(parity);
      PageWalk w;
      w.start(meta, P.cache_seqlens, P.max_blocks);
      int n = 0, seg = 0;
      bool ok = true;
      while (w.valid && ok) {
        if (w.first()) {
          // Both issuers wait for every segment's Q, also for a segment they
          // own no page of: a parity wait on a barrier that may still be a
          // phase behind would otherwise pass early.
          ok = mbar_wait(bar(kBarQFull), seg & 1, abort_flag);
          if (!ok) break;
          ++seg;
        }
        if ((n & 1) == parity) {
          if (n >= 2) {
            ok = mbar_wait(bar(kBarSFree + parity), ((n >> 1) - 1) & 1, abort_flag);
            if (!ok) break;
          }
          const int st = n % kStages;
          ok = mbar_wait(bar(kBarFull + st), (n / kStages) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after_sync();
          const uint64_t koff = static_cast<uint64_t>((st * kKStage) >> 4);
#pragma unroll
          for (int c = 0; c < 3; ++c) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              umma_bf16_ts(d, tmem + kTmemQ + 32 * c + 8 * ks,
                           d_klat + koff + static_cast<uint64_t>((c * kKChunk + ks * 32) >> 4), kIdescQK,
                           (c | ks) != 0);
            }
          }
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_bf16(d, d_qlat + static_cast<uint64_t>((ks * 32) >> 4),
                      d_klat + koff + static_cast<uint64_t>((3 * kKChunk + ks * 32) >> 4), kIdescQK, 1);
#pragma unroll
          for (int ks = 0; ks < 2; ++ks)
            umma_bf16(d, d_qrope + static_cast<uint64_t>((ks * 32) >> 4),
                      d_krope + koff + static_cast<uint64_t>((ks * 32) >> 4), kIdescQK, 1);
          umma_commit(bar(kBarSFull + parity));
        }
        // Q may be replaced once every QK of this segment is done: two arrivals,
        // one per issuer, or both from the issuer of a single-page segment.  An
        // issuer that owns no page of a segment does not arrive for it, so no
        // arrival can ever count towards the wrong segment.
        if (w.last()) {
          if (w.p_end - w.p_begin > 1) {
            umma_commit(bar(kBarQEmpty));
          } else if ((n & 1) == parity) {
            umma_commit(bar(kBarQEmpty));
            umma_commit(bar(kBarQEmpty));
          }
        }
        ++n;
        w.advance();
      }
      if (!ok) raise_status(P.status, kStatusTimeout);
      umma_commit(bar(kBarDone));
      drain_wait(bar(kBarDone), 0);
    }
    __syncwarp();
  }
  } else if (warp >= kFirstSoftmaxWarp) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ================================================= softmax + epilogue
    // Warp (quad, half) owns the 16 rows 32*quad + 16*half + [0,16) -- lanes of
    // its tensor-memory quadrant -- over all 64 tokens of every page.  Lane l
    // holds row (l & 15) and tokens 32*(l >> 4) + [0,32): a row's two halves sit
    // in lanes l and l^16, so its max and sum need one shuffle and no other warp.
    const int quad = warp & 3;
    const int sw = warp - kFirstSoftmaxWarp;  // softmax warp index: the exchange slot region it owns
    const int half = sw >> 2;                 // which 16 lanes of the quadrant
    const int lane_i = static_cast<int>(lane);
    const int row = 32 * quad + 16 * half + (lane_i & 15);
    const int tok0 = 32 * (lane_i >> 4);      // this lane's first token of a page
    const uint32_t lane_off = static_cast<uint32_t>(32 * quad + 16 * half) << 16;
    const bool leader = (sw == 0 && lane == 0);
    const uint32_t peer_xempty = cluster_map(bar(kBarXEmpty), peer);

    // row -> (query position, head)
    const int jj = row / P.heads_per_kv;
    const int hh = row - jj * P.heads_per_kv;
    const int j = tile * P.q_per_tile + jj;
    const int h = g * P.heads_per_kv + hh;
    const bool row_live = (row < rows_valid) && (j < P.s_q);
    // A warp whose 16 rows hold no query position keeps the hand-offs but
    // skips the peer's partial (none is sent for those rows).  Its scores are
    // never written out; rows are independent in every step, so whatever they
    // hold cannot reach a live row.
    const bool warp_live = 32 * quad + 16 * half < rows_live;
    const int rows_total = P.s_q * P.h_q;
    const int row_in_seq = j * P.h_q + h;
    // Scores stay in raw units (q.k); scale*log2(e) is applied inside the exp2
    // argument, and the lazy-rescale threshold is converted to raw units.
    const float c_log2 = P.scale_log2;
    const float rescale_raw = kRescaleThreshold / c_log2;

    PageWalk w;
    w.start(meta, P.cache_seqlens, P.max_blocks);
    float m_run = -INFINITY, l_run = 0.f;
    int lim = 0;
    int n = 0;
    int groups = 0;  // P hand-offs to the PV warp so far (two on pages with a low-part pass)
    int lo_check = -1;  // page whose low-part decision is still open, or -1
    uint32_t lo[16];    // that page's low part of P (zero if this warp did not ask)
    bool ok = true;
    while (ok && w.valid) {
      if (w.first()) {
        const int L = __ldg(P.cache_seqlens + w.i);
        lim = min(P.causal ? L - P.s_q + j + 1 : L, L);
        m_run = -INFINITY;
        l_run = 0.f;
      }
      // ======== page n: own partial S out of tensor memory (the sender warps
      // quantise and send the same partial to the peer meanwhile)
      const int sb = n & 1;
      const int slot = n % kXSlots;
      if (leader) mbar_arrive_expect_tx(bar(kBarXFull + slot), static_cast<uint32_t>(rows_live) * kXRowBytes);
      ok = mbar_wait(bar(kBarSFull + sb), (n >> 1) & 1, abort_flag);
      if (!ok) break;
      tc_fence_after_sync();
      float x[32];
      {
        uint32_t s[32];
        tmem_ld16x2_32(tmem + lane_off + kTmemS + 64u * sb, s);
        tmem_wait_ld(s);
#pragma unroll
        for (int c = 0; c < 32; ++c) x[c] = __uint_as_float(s[c]);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarSFree + sb));

      // ======== add the peer's partial
      ok = mbar_wait(bar(kBarXFull + slot), (n / kXSlots) & 1, abort_flag);
      if (!ok) break;
      if (warp_live) {
        const uint8_t* xr = gbase + kOffX + slot * kXSlot;
        const float sc = *reinterpret_cast<const float*>(xr + x_scale(sw, lane_i));
        const uint64_t sc2 = f2(sc, sc), nbase2 = f2(-kQuantBase, -kQuantBase);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = *reinterpret_cast<const uint4*>(xr + x_chunk(sw, lane_i, k));
          const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 8 * k + 2 * e;
            const uint64_t q = f2_add(f2(__uint_as_float(__byte_perm(wv[e], kQuantHi, 0x7610)),
                                         __uint_as_float(__byte_perm(wv[e], kQuantHi, 0x7632))),
                                      nbase2);
            f2_split(f2_fma(q, sc2, f2(x[c], x[c + 1])), x[c], x[c + 1]);
          }
        }
      }

      // The slot has been read: the last of the 8 softmax warps to finish
      // returns it to the peer's senders.  Each warp's fence orders its lanes'
      // loads (after the warp barrier) before its count; the last warp's fence
      // orders all of them before its remote arrive.
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        if (atomicAdd(xread_cnt + slot, 1u) == 7u) {
          xread_cnt[slot] = 0u;
          __threadfence_block();
          mbar_arrive_cluster_relaxed(peer_xempty + 8u * static_cast<uint32_t>(slot));
        }
      }

      // ======== online softmax
      const int t0 = w.p * kPage + tok0;
      if (t0 + 32 > lim) {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (t0 + c >= lim) x[c] = -INFINITY;
      }
      float mx4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) mx4[u] = x[u];
#pragma unroll
      for (int c = 4; c < 28; c += 8) {
#pragma unroll
        for (int u = 0; u < 4; ++u) mx4[u] = fmax3(mx4[u], x[c + u], x[c + 4 + u]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) mx4[u] = fmaxf(mx4[u], x[28 + u]);
      const float mx_lane = fmaxf(fmax3(mx4[0], mx4[1], mx4[2]), mx4[3]);
      const float mx = fmaxf(mx_lane, __shfl_xor_sync(0xffffffffu, mx_lane, 16));  // the row's other 32 tokens
      float alpha = 1.f;
      {
        const float m_new = fmaxf(m_run, mx);
        if (m_new > m_run + rescale_raw) {
          alpha = ex2_approx((m_run - m_new) * c_log2);  // 0 when m_run = -inf
          m_run = m_new;
        }
      }
      const float neg_mc = (m_run == -INFINITY) ? 0.f : -m_run * c_log2;
      uint32_t pk[16];
      float rsum;
      {
        const uint64_t c2 = f2(c_log2, c_log2), nmc2 = f2(neg_mc, neg_mc);
        uint64_t sum2[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) sum2[u] = f2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          float a0, a1;
          f2_split(f2_fma(f2(x[2 * c], x[2 * c + 1]), c2, nmc2), a0, a1);
          const float e0 = ex2_approx(a0);
          const float e1 = ex2_approx(a1);
          sum2[c & 3] = f2_add(sum2[c & 3], f2(e0, e1));
          pk[c] = pack_bf16x2(e0, e1);
        }
        float sum8[8];
#pragma unroll
        for (int u = 0; u < 4; ++u) f2_split(sum2[u], sum8[2 * u], sum8[2 * u + 1]);
        rsum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      }
      l_run = l_run * alpha + rsum;  // this lane's 32 tokens; the row sum adds lane l^16's
      // Does a weight of this warp's rows exceed a third of its row's sum so
      // far?  (-inf lanes give 0, NaN compares false.)
      const bool want_lo =
          __any_sync(0xffffffffu, ex2_approx(fmaf(mx_lane, c_log2, neg_mc)) * kLoRatio >
                                      l_run + __shfl_xor_sync(0xffffffffu, l_run, 16));

      // The previous page's low part, if any warp asked for it: once its bf16
      // part's PV is complete (it read the P buffer), every warp stores its own
      // low part (zero where it did not ask) and the PV warp adds P_lo V to O.
      if (groups > 0) {
        ok = mbar_wait(bar(kBarOFull), (groups - 1) & 1, abort_flag);
        if (!ok) break;
        if (lo_check >= 0) {
          ok = lo_pass(bar(kBarPFull), bar(kBarOFull), lo_flag, lo_check, groups, tmem + lane_off + kTmemP, lo,
                       abort_flag);
          if (!ok) break;
          lo_check = -1;
        }
        tc_fence_after_sync();
      }
      tmem_st16x2(tmem + lane_off + kTmemP, pk);
      const bool rescale_o = !w.first() && alpha != 1.f;
      if (__any_sync(0xffffffffu, rescale_o)) rescale_o_half(tmem + lane_off + kTmemO, alpha);
      tmem_wait_st();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (want_lo) atomicMax(const_cast<int*>(lo_flag) + (n & 1), n + 1);
        mbar_arrive(bar(kBarPFull));
      }
      ++groups;
      // This page's low part is decided once every warp has handed P over:
      // before the next P store, or right here at the end of a segment.
      if (want_lo) {
        const uint64_t c2 = f2(c_log2, c_log2), nmc2 = f2(neg_mc, neg_mc);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          // the bf16 rounding error of the pair (same weights as above), itself rounded to bf16
          float a0, a1, r0, r1;
          f2_split(f2_fma(f2(x[2 * c], x[2 * c + 1]), c2, nmc2), a0, a1);
          f2_split(f2_sub(f2(ex2_approx(a0), ex2_approx(a1)),
                          f2(__uint_as_float(pk[c] << 16), __uint_as_float(pk[c] & 0xffff0000u))),
                   r0, r1);
          lo[c] = pack_bf16x2(r0, r1);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) lo[c] = 0u;
      }
      lo_check = n;
      if (w.last()) {
        ok = lo_pass(bar(kBarPFull), bar(kBarOFull), lo_flag, lo_check, groups, tmem + lane_off + kTmemP, lo,
                     abort_flag);
        if (!ok) break;
        lo_check = -1;
      }

      // ======== epilogue at the end of a segment
      if (w.last()) {
        const float l_tot = l_run + __shfl_xor_sync(0xffffffffu, l_run, 16);
        ok = mbar_wait(bar(kBarOFull), (groups - 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after_sync();
        const int nsplit = __ldg(P.num_splits + w.i + 1) - __ldg(P.num_splits + w.i);
        const bool direct = (nsplit == 1);
        const float inv_l = (l_tot > 0.f) ? 1.f / l_tot : 0.f;
        const float lse = (l_tot > 0.f) ? (m_run * c_log2 + log2f(l_tot)) * 0.69314718055994531f : -INFINITY;
        const int64_t oslot = static_cast<int64_t>(__ldg(P.num_splits + w.i)) + w.k;
        const uint32_t live = __ballot_sync(0xffffffffu, row_live);
        if (direct)
          write_o_rows(tmem + lane_off + kTmemO, inv_l,
                       static_cast<__nv_bfloat16*>(P.out) + static_cast<int64_t>(w.i) * rows_total * kDimV, nullptr,
                       256 * static_cast<int>(rank), row_in_seq, live);
        else
          write_o_rows(tmem + lane_off + kTmemO, inv_l, nullptr,
                       static_cast<float*>(P.ws_o) + oslot * rows_total * kDimV, 256 * static_cast<int>(rank),
                       row_in_seq, live);
        if (row_live && rank == 0 && lane_i < 16) {
          if (direct)
            P.lse[(static_cast<int64_t>(w.i) * P.h_q + h) * P.s_q + j] = lse;
          else
            P.ws_lse[oslot * rows_total + row_in_seq] = lse;
        }
        tc_fence_before_sync();
      }
      ++n;
      w.advance();
    }
    if (!ok) raise_status(P.status, kStatusTimeout);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsStage));
    // ================================================= Q staging + exchange sending
    // Warps 0-3 stage each segment's Q -- this CTA's 256 latent dims of each
    // row: [0, 192) into tensor memory as bf16 pairs, [192, 256) into shared
    // memory (128B swizzle, K-major).  Per page, thread `row` reads its row's
    // 64 partial scores out of tensor memory, quantises each 32-token half and
    // writes it with st.async into the peer's receive slot, at the place of
    // the peer softmax thread that owns the row, once the peer has returned
    // that slot: they, not the softmax warps, do the quantisation and absorb
    // the SM-to-SM link's back-pressure.  A segment's Q is staged once the
    // previous segment's QKs are done (warp 0 also starts the TMA load of its
    // 32 rope dims then), and before its first page can be sent.
    const int quad = warp & 3;
    const int row = 32 * quad + static_cast<int>(lane);
    const uint32_t lane_off = static_cast<uint32_t>(32 * quad) << 16;
    const int jj = row / P.heads_per_kv;
    const int hh = row - jj * P.heads_per_kv;
    const int j = tile * P.q_per_tile + jj;
    const int h = g * P.heads_per_kv + hh;
    const bool row_live = (row < rows_valid) && (j < P.s_q);
    const __nv_bfloat16* qbase = static_cast<const __nv_bfloat16*>(P.q);
    const uint32_t peer_x = cluster_map(base + kOffX, peer);
    const uint32_t peer_xfull = cluster_map(bar(kBarXFull), peer);
    // A warp with no live row writes nothing into the peer's slot, so it does
    // not wait for the slot's credit either: the credit's phases follow the
    // warps that send, and a waiter that fell two phases behind them would
    // wait on the wrong phase.
    const bool sends = __any_sync(0xffffffffu, row_live);
    const int dim_rope = 512 + 32 * static_cast<int>(rank);
    int lim = 0;  // visible tokens of this row in the current sequence

    auto load32 = [&](const uint8_t* src, uint32_t (&r)[32]) {
      if (row_live) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 v = ld_global_nc_v4(src + 16 * k);
          r[4 * k + 0] = v.x;
          r[4 * k + 1] = v.y;
          r[4 * k + 2] = v.z;
          r[4 * k + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) r[k] = 0u;
      }
    };
    PageWalk wq, w;
    wq.start(meta, P.cache_seqlens, P.max_blocks);
    w = wq;
    int qseg = 0;  // segments whose Q has been staged
    bool ok = true;
    auto stage_q = [&]() -> bool {
      const uint8_t* src = reinterpret_cast<const uint8_t*>(
          qbase + ((static_cast<int64_t>(wq.i) * P.s_q + j) * P.h_q + h) * kDimQK + 256 * rank);
      uint32_t q0[32], q1[32];
      load32(src, q0);
      load32(src + 128, q1);
      if (!mbar_wait(bar(kBarQEmpty), (qseg & 1) ^ 1, abort_flag)) return false;
      if (warp == 0 && lane == 0) {
        mbar_arrive_expect_tx(bar(kBarQFull), static_cast<uint32_t>(rows_valid) * 64u);
        tma_load_4d(base + kOffQR, &q_rope, bar(kBarQFull), dim_rope, g * P.heads_per_kv, tile * P.q_per_tile,
                    wq.i);
      }
      tc_fence_after_sync();
      tmem_st32(tmem + lane_off + kTmemQ, q0);
      tmem_st32(tmem + lane_off + kTmemQ + 32, q1);
      // the second half in one round of loads
      load32(src + 256, q0);
      load32(src + 384, q1);
      tmem_st32(tmem + lane_off + kTmemQ + 64, q0);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        *reinterpret_cast<uint4*>(gbase + kOffQL + row * 128 + ((k ^ (row & 7)) << 4)) =
            make_uint4(q1[4 * k], q1[4 * k + 1], q1[4 * k + 2], q1[4 * k + 3]);
      fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarQFull));
      ++qseg;
      wq.next_segment();
      return true;
    };
    // The warps poll: the next page is sent as soon as its S is ready (the
    // peer's softmax waits for it); otherwise a segment's Q is staged once the
    // previous segment's QKs are done (the next segment's first QK waits for
    // it, and its K pages are still in flight).  A send waits only for the
    // peer's progress on earlier pages, so this order cannot deadlock.  Each
    // decision is lane 0's, broadcast, so the warp stays converged.
    int n = 0;
    long long t_idle = clock64();
    while (ok && (w.valid || wq.valid)) {
      const bool s_ready =
          __shfl_sync(0xffffffffu, (w.valid && mbar_test(bar(kBarSFull + (n & 1)), (n >> 1) & 1)) ? 1 : 0, 0) != 0;
      if (!s_ready && __shfl_sync(0xffffffffu, (wq.valid && mbar_test(bar(kBarQEmpty), (qseg & 1) ^ 1)) ? 1 : 0, 0)) {
        ok = stage_q();
        t_idle = clock64();
        continue;
      }
      if (!s_ready) {
        if (w.valid) mbar_try_wait_for(bar(kBarSFull + (n & 1)), (n >> 1) & 1, 200);
        else mbar_try_wait_for(bar(kBarQEmpty), (qseg & 1) ^ 1, 200);
        int give_up = (*abort_flag || clock64() - t_idle > kWaitTimeoutCycles) ? 1 : 0;
        if (__shfl_sync(0xffffffffu, give_up, 0)) {
          *abort_flag = 1;
          ok = false;
        }
        continue;
      }
      t_idle = clock64();
      // ---- page n: this CTA's partial S of row `row`, quantised per 32 tokens
      if (w.first()) {
        const int L = __ldg(P.cache_seqlens + w.i);
        lim = min(P.causal ? L - P.s_q + j + 1 : L, L);
      }
      const int sb = n & 1;
      ok = mbar_wait(bar(kBarSFull + sb), (n >> 1) & 1, abort_flag);
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t s0[32], s1[32];
      tmem_ld32(tmem + lane_off + kTmemS + 64u * sb, s0);
      tmem_ld32(tmem + lane_off + kTmemS + 64u * sb + 32u, s1);
      tmem_wait_ld2(s0, s1);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarSFree + sb));
      uint32_t enc[2][16];
      float scl[2];
#pragma unroll
      for (int th = 0; th < 2; ++th) {
        float a[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) a[c] = __uint_as_float(th ? s1[c] : s0[c]);
        const int t0 = w.p * kPage + 32 * th;
        if (t0 + 32 > lim) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (t0 + c >= lim) a[c] = 0.f;
        }
        float amax8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) amax8[u] = fabsf(a[u]);
#pragma unroll
        for (int c = 8; c < 32; ++c) amax8[c & 7] = fmaxf(amax8[c & 7], fabsf(a[c]));
        const float amax = fmaxf(fmaxf(fmaxf(amax8[0], amax8[1]), fmaxf(amax8[2], amax8[3])),
                                 fmaxf(fmaxf(amax8[4], amax8[5]), fmaxf(amax8[6], amax8[7])));
        const float inv = (amax > 0.f) ? __fdividef(kQuantMax, amax) : 0.f;
        const uint64_t inv2 = f2(inv, inv), base2 = f2(kQuantBase, kQuantBase);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float t0f, t1f;
          f2_split(f2_fma(f2(a[2 * e], a[2 * e + 1]), inv2, base2), t0f, t1f);
          enc[th][e] = __byte_perm(__float_as_uint(t0f), __float_as_uint(t1f), 0x5410);
        }
        scl[th] = amax * (1.0f / kQuantMax);
      }
      const int slot = n % kXSlots;
      if (sends && n >= kXSlots) {
        // the peer has read page n - kXSlots out of the slot page n goes to
        ok = mbar_wait<true>(bar(kBarXEmpty + slot), ((n / kXSlots) - 1) & 1, abort_flag);
        if (!ok) break;
      }
      const uint32_t dst = peer_x + static_cast<uint32_t>(slot * kXSlot);
      const uint32_t xb = peer_xfull + 8u * static_cast<uint32_t>(slot);
      // the peer's softmax warp (quad, lane >> 4) owns this row; its lanes
      // (lane & 15) and (lane & 15) + 16 take tokens [0, 32) and [32, 64)
      const int rsw = quad + 4 * static_cast<int>(lane >> 4);
#pragma unroll
      for (int th = 0; th < 2; ++th) {
        if (!row_live) break;  // rows past the tile's query positions are not exchanged
        const int rl = static_cast<int>(lane & 15) + 16 * th;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          st_async_v4(dst + x_chunk(rsw, rl, k), enc[th][4 * k], enc[th][4 * k + 1], enc[th][4 * k + 2],
                      enc[th][4 * k + 3], xb);
        st_async_b32(dst + x_scale(rsw, rl), __float_as_uint(scl[th]), xb);
      }
      ++n;
      w.advance();
    }
    if (!ok) {
      raise_status(P.status, kStatusTimeout);
      // let the last rope load land before this CTA can exit
      if (warp == 0 && lane == 0 && qseg > 0) drain_wait(bar(kBarQFull), (qseg - 1) & 1);
    }
  }

  // ---- teardown: everyone is done with tensor memory and with the peer
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 5) {
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
  // Programmatic stream serialisation: the CTAs start (tensor memory,
  // barriers, cluster sync) while the scheduler kernel before them finishes.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * num_parts, row_tiles, p.h_kv);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_decode_kernel, q_rope, k_lat, k_rope, p);
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
