// Step 3: split-KV absorbed-MLA partial attention on the sm_103a tensor cores.
//
// "[ROCm][MLA][DCP] Support causal multi-token verification", Implementation
// item 3: each rank attends its local KV and emits unreduced partial outputs with
// base-2 max/sum statistics. "Context Parallel Guide (PCP & DCP)", "How it works"
// item 4: the FP8 cache carries one per-tensor scale.
//
// Work item = (rank, sequence, split, 128-row tile of the sequence's qlen*H query
// rows, j-major). Each work item runs on a CLUSTER OF TWO CTAs (one per SM):
//
//   * One 128-row fp32 accumulator over all 512 value dims would fill the SM's
//     whole tensor memory, leaving no room for the scores. So the value dims are
//     split: CTA c accumulates O[:, 256c : 256c+256] (256 TMEM columns).
//   * Both CTAs need the full scores. Instead of computing them twice, the 576
//     q/k dims are split too: CTA0 computes the partial score x0 over dims
//     [0, 256), CTA1 x1 over dims [256, 576) (log2 units). Shared memory across
//     the pair is slow (about 18 bytes per cycle per SM each way, measured), so a
//     CTA does not send x itself: for each (row, 32-token half) it sends its own
//     maximum m_c and the factors E_c = 2^(x_c - m_c) in f16 (scaled by 2^14, so
//     values down to 2^-28 keep 11 bits), and keeps the same f16 words. Both CTAs
//     then form bit-identical weights
//         p = E_own * E_peer * 2^(m_own + m_peer - M)
//     (the f16 product is exact in f32), where M is the running reference of the
//     row. The tile bound max_half(m_own + m_peer) is an upper bound of the true
//     maximum, but it can lie far above it when the two partial scores of the row
//     disagree (a token large on one span only, another on the other). So M is
//     raised only when the bound passes M + 15, and then set 7 below the bound: p
//     stays below 2^15 (finite in f16), and the tile's largest weight stays in f16's
//     normal range while the bound overestimates the true maximum by up to 21
//     binades. Relative error of p and l from the two f16 factors: at most 2^-10.
//   * CTA c stages dims [256c, 256c + 256 + 64c) of every token: its q.k slice,
//     which also holds its value slice.
//   * A thread issuing straight-line tcgen05.mma gets about one instruction per
//     55 (N=64) to 130 (N=256) cycles; branches or arithmetic between them were
//     measured to double that. The whole q.k contraction is one straight-line
//     chain (q from tensor memory), and P.V has its own issuing thread.
//   * The per-tile softmax work is split in two stages on different warps. The front
//     warps turn the scores of tile i into factors and send them; they keep no state
//     across tiles (the factors are relative to the half's own maximum). The back
//     warps then finish tile i with the peer's factors: the running reference, P,
//     and l. So the exchange latency and the front of the next tile overlap the back
//     of the current one, and the front runs up to two tiles ahead (the exchange and
//     own-factor buffers are double-buffered). P.V starts as soon as P is written.
//
// Per CTA (704 threads; 80 registers each: the six warps of a sub-partition share its
// 16K registers):
//   warps 0-7   front: warp w owns rows 32*(w%4) .. +31 (TMEM lane quarter) and token
//               half w/4 of every 64-token tile; Q into TMEM at the start; S -> own
//               f16 factors and the half maximum -> the peer's exchange slot
//               (st.async) and the local own-factor buffer.
//   warps 8-15  back: the same rows and halves. One wait covers the peer's factors,
//               the local front warps' factors and maxima, and the completion of the
//               previous tile's P.V (all are arrivals on the slot's barrier). Lazy
//               online softmax, P (16-bit) into TMEM, l.
//   epilogue    all 16 warps: 64 O columns each of their rows.
//   warps 16-19 KV producers: 16-byte loads of the paged cache rows (subpage ids
//               from the metadata, bounds-checked), FP8 E4M3 -> f16 conversion,
//               stores into 128-byte-swizzled K-major tiles of a 3-stage ring.
//               FP8 keeps two tiles in flight (registers + cp.async staging in
//               shared memory), so a freed stage only waits for the conversion.
//   warp 20     TMEM allocation; issues S = Q[tmem] . K_tile^T (M=128, N=64, all
//               of this CTA's dims).
//   warp 21     issues O += P[tmem] . V_tile (M=128, N=256, V read MN-major from
//               the same swizzled tile as K).
//   The issuing warps run converged and one elected lane issues each tcgen05
//   instruction, so its operands are warp-uniform values.
// TMEM columns: O [0,256), S [256,320), P [320,352), Q [352,512) (CTA1: five
// 64-dim atoms, CTA0: four). The FP8-cache path computes in f16 (E4M3 -> f16
// is exact; q is BF16 -> f16, exact in f16's normal range; |q| > 65504 sets
// DCP_STATUS_Q_RANGE); the BF16-cache path computes in bf16. Accumulation is
// fp32 throughout.
//
// Every wait is bounded (DCP_STATUS_TIMEOUT and an orderly exit: all roles stop,
// in-flight MMAs are drained, TMEM is freed). A wait checks once with a plain
// mbarrier.try_wait, then sleeps in try_wait with a suspend-time hint. Nothing traps.
//
// Work items reach clusters longest first (order_kernel, below), so that items of
// very different lengths finish together.
#include <climits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "sm103.cuh"

namespace dcpmla {
namespace {

using namespace sm103;

constexpr int kTileN = 64;     // tokens per KV tile
constexpr int kRows = 128;     // query rows per tile (MMA M)
constexpr int kStages = 3;     // KV ring depth
constexpr int kMaxAtoms = 5;   // 64-dim swizzle atoms staged per CTA (CTA1: 320 dims)
constexpr int kAtomBytes = kTileN * 128;
constexpr int kStageBytes = kMaxAtoms * kAtomBytes;
// factor exchange slot: E as f16 [half 2][group 4][row 128][8 values], m as f32 [half][row]
constexpr int kXchEBytes = 2 * 4 * kRows * 16;
constexpr int kXchSlotBytes = kXchEBytes + 2 * kRows * 4;
constexpr int kXchSlots = 2;
constexpr int kMOwnBufs = 2;  // own half maxima, by tile mod 2 (the front warps write tile
                              // t+2 once the back warps have finished tile t)
constexpr int kMOwnBytes = kMOwnBufs * 2 * kRows * 4;   // [tile%2][half][row] f32
constexpr int kLCombBytes = 2 * kRows * 4;              // [half][row] f32, epilogue
constexpr int kEInvBytes = kRows * 4;                   // [row] f32, epilogue output scale
constexpr int kEPrevBytes = 2 * 2 * 4 * kRows * 16;  // own f16 factors, as sent:
                                                     // [tile%2][half][group 4][row][8]
// FP8 producer staging: each producer thread's 16-byte chunks of one tile (the
// tile after next), [chunk][thread], written by cp.async
constexpr int kRawBytes = kMaxAtoms * 2 * 128 * 16;
constexpr int kFrontWarps = 8;   // warps 0-7: scores -> own factors -> peer
constexpr int kBackWarps = 8;    // warps 8-15: both CTAs' factors -> P, running reference
constexpr int kSoftWarps = kFrontWarps + kBackWarps;
constexpr int kProdWarp0 = 16;
constexpr int kMmaWarpS = 20;
constexpr int kMmaWarpP = 21;
constexpr int kThreads = 22 * 32;
constexpr uint32_t kColO = 0, kColS = 256, kColP = 320, kColQ = 352;
constexpr uint32_t kTmemCols = 512;
// Lazy reference: M is raised only when the tile bound passes M + kRaiseAbove, and
// then set kRefBelow under the bound. P <= 2^(bound - M) <= 2^15 stays finite in f16,
// and right after a raise P <= 2^7, so the largest weight of the tile keeps full f16
// precision while the bound overestimates the true maximum by up to 21 binades.
constexpr float kRaiseAbove = 15.0f;
constexpr float kRefBelow = 7.0f;
constexpr float kFactorLog2 = 14.0f;       // factors carry 2^14: E down to 2^-28 stays normal in f16
constexpr uint64_t kTimeoutNs = 4000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

// barrier slots
enum {
  kBarKvFull = 0,
  kBarKvEmpty = kBarKvFull + kStages,  // count 2: score chain, P.V
  kBarSFull = kBarKvEmpty + kStages,   // score chain committed
  kBarSFree,                           // count 8: softmax warps read S
  kBarPFull,                           // count 8: P written
  kBarODone,                           // P.V completed
  kBarQFull,                           // count 8
  kBarXFull,                           // [2] count 10: the peer's factors are in my slot,
                                       // the 8 local warps wrote their half maxima and the
                                       // previous tile's P.V completed
  kBarXFree = kBarXFull + kXchSlots,   // [2] count 8: the peer consumed what I wrote
  kBarEFree = kBarXFree + kXchSlots,   // [2] count 8: the local back warps consumed the
                                       // own factors and maxima of that slot
  kBarLComb = kBarEFree + kXchSlots,   // count 8: epilogue l halves written
  kBarEpi,                             // count 8: the output scale of every row written
  kBarDrainS,
  kBarDrainP,
  kNumBars
};

constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + kStages * kStageBytes +
                              kXchSlots * kXchSlotBytes + kMOwnBytes + kLCombBytes +
                              kEInvBytes + kEPrevBytes + kRawBytes + kNumBars * 8 + 16;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

struct Params {
  const uint16_t* q;
  const uint8_t* kv;
  const float* kv_scale;
  const int32_t* row_len;
  const int32_t* page_ids;
  const int32_t* split_beg;
  const int32_t* split_end;
  float* part_o;
  float* part_m;
  float* part_l;
  uint32_t* status;
  const int32_t* item_order;  // cluster -> work item (longest first), or null: natural order
  const int32_t* n_live;      // clusters with an item in item_order (the rest exit at once)
  // packed epilogue (one split): the all-to-all send buffers [rank][G][cw words] get the
  // BF16 output and the LSE words instead of part_o/m/l (null: the fp32 partials)
  uint16_t* send;
  int64_t send_cw;
  int G;
  float softmax_scale;
  int batch, qlen, H, num_splits, subpage, max_pages, n_row_tiles;
  int64_t pool_rows;  // rows of one rank's pool: num_blocks * block_size
  // The failure path's test: hold_q = 1 withholds the softmax warps' arrivals on the q
  // barrier, so the score issuer's wait for q runs out after q_wait_ns and the kernel
  // stops in order (DCP_STATUS_TIMEOUT). 0 and the 4 s limit in every other call.
  int hold_q;
  uint64_t q_wait_ns;
};

struct Shared {
  uint8_t* stages;
  uint8_t* xch;   // kXchSlots slots
  float* mown;    // own half maxima per tile
  float* lcomb;   // epilogue l halves
  float* einv;    // epilogue output scale per row
  uint4* eprev;   // own factors (f16, as sent) of the last two tiles
  uint8_t* raw;   // FP8 producer staging
  uint64_t* bars;
  uint32_t* tmem_slot;
  int* abort_flag;
};

__device__ __forceinline__ Shared carve(unsigned char* raw) {
  Shared s;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  s.stages = base;
  s.xch = base + kStages * kStageBytes;
  s.mown = reinterpret_cast<float*>(s.xch + kXchSlots * kXchSlotBytes);
  s.lcomb = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(s.mown) + kMOwnBytes);
  s.einv = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(s.lcomb) + kLCombBytes);
  s.eprev = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(s.einv) + kEInvBytes);
  s.raw = reinterpret_cast<uint8_t*>(s.eprev) + kEPrevBytes;
  s.bars = reinterpret_cast<uint64_t*>(s.raw + kRawBytes);
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.bars + kNumBars);
  s.abort_flag = reinterpret_cast<int*>(s.tmem_slot + 1);
  return s;
}

// Bounded wait on an mbarrier phase. Checking a phase that has already
// completed was measured at ~67 cycles with a plain try_wait and ~121 with a
// suspend-time hint, while a waiter that has to sleep notices the completion
// ~170 cycles after the arrive with the hint and ~280 without. So the first
// check is a plain try_wait, and the slow path repeats hinted try_waits; between
// them it checks the abort flag and gives up after limit_ns (raising the abort
// flag and DCP_STATUS_TIMEOUT).
__device__ __noinline__ bool wait_phase_slow(uint32_t a, uint32_t parity, int* abort_flag,
                                             uint32_t* status, bool cluster_acquire,
                                             uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (cluster_acquire ? mbar_wait_sleep_cluster(a, parity) : mbar_wait_sleep(a, parity))
      return true;
    if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *reinterpret_cast<volatile int*>(abort_flag) = 1;
      raise_status(status, DCP_STATUS_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, int* abort_flag,
                                           uint32_t* status, bool cluster_acquire,
                                           uint64_t limit_ns = kTimeoutNs) {
  const uint32_t a = smem_u32(bar);
  if (cluster_acquire ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity)) return true;
  return wait_phase_slow(a, parity, abort_flag, status, cluster_acquire, limit_ns);
}

// wait_phase for a whole converged warp, with a warp-uniform result (the
// elect.sync of the tcgen05 issue that follows needs every lane).
__device__ __forceinline__ bool wait_uniform(uint64_t* bar, uint32_t parity, int* abort_flag,
                                             uint32_t* status, uint64_t limit_ns = kTimeoutNs) {
  return __all_sync(0xffffffffu, wait_phase(bar, parity, abort_flag, status, false, limit_ns));
}

struct Item {
  int k, b, s, t;
  int qr0, rows_valid;
  int t_start, t_end, n_tiles;
  bool bad_split;  // the split bounds were outside [0, MP] (the item then covers nothing)
};

// Work item `item` (natural order: rank, sequence, split, row tile, the row tile
// fastest) with its tile range.
__device__ __forceinline__ Item decode_item(const Params& p, int item) {
  Item it;
  it.bad_split = false;
  int rest = item;
  it.t = rest % p.n_row_tiles;
  rest /= p.n_row_tiles;
  it.s = rest % p.num_splits;
  rest /= p.num_splits;
  it.b = rest % p.batch;
  it.k = rest / p.batch;
  const int qrows = p.qlen * p.H;
  it.qr0 = it.t * kRows;
  it.rows_valid = min(kRows, qrows - it.qr0);
  const int R = p.batch * p.qlen;
  const int j_lo = it.qr0 / p.H;
  const int j_hi = (it.qr0 + it.rows_valid - 1) / p.H;
  int maxL = 0;
  for (int j = j_lo; j <= j_hi; ++j)
    maxL = max(maxL, p.row_len[(int64_t)it.k * R + (int64_t)it.b * p.qlen + j]);
  const int64_t sb = ((int64_t)it.k * p.batch + it.b) * p.num_splits + it.s;
  int beg = p.split_beg[sb], end = p.split_end[sb];
  if (beg < 0 || end < beg || end > p.max_pages) {  // the status is raised once, by the kernel
    it.bad_split = true;
    beg = end = 0;
  }
  it.t_start = beg * p.subpage;
  it.t_end = min(end * p.subpage, maxL);
  it.n_tiles = it.t_end > it.t_start ? (it.t_end - it.t_start + kTileN - 1) / kTileN : 0;
  return it;
}

// 2^x on the MUFU unit (ex2.approx, flush-to-zero); x <= 8 here and results
// below 2^-126 only ever meet other tiny weights.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Four E4M3 codes -> two f16x2 words (exact): the hardware conversion applied to
// both 16-bit halves of the word (byte k of x becomes half k of the result).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t x, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}

// ----------------------------------------------------------------- producers
// Each producer thread owns fixed tokens of every tile and one 16-byte column
// of every atom: FP8 -> tokens tk0 and tk0+32 (tk0 = ct/4), 16 dims at
// quarter ct%4 (two f16 chunks out); BF16 -> tokens tk0 + 16j (tk0 = ct/8),
// 8 dims at chunk ct%8. A warp then covers 8 (or 4) consecutive tokens of one
// atom: contiguous global reads per token and shared stores that fill whole
// 128-byte swizzled rows. Row addresses are formed once per token per tile, so
// the unrolled load/store code is short (it competes for instruction cache
// with the softmax warps of the same SM).
template <bool kFp8, int kAtoms>
struct Producer {
  static constexpr int kElem = kFp8 ? 1 : 2;
  static constexpr int kD0 = 256 * (kAtoms - 4);  // first staged dim: 0 (CTA0) or 256 (CTA1)
  static constexpr int kToks = kFp8 ? 2 : 4;       // tokens per thread per tile
  static constexpr int kTokStride = kFp8 ? 32 : 16;
  static constexpr int kLoads = kAtoms * kToks;

  const Params& p;
  const Shared& sh;
  const Item& it;
  int lg_sub, tk0;
  uint32_t col;   // byte offset of this thread's 16 bytes inside an atom row (global)
  uint32_t soff0; // swizzled smem offset of this thread's first output chunk, token tk0
  int64_t pool_pages;
  const uint8_t* pool;
  const int32_t* pages;
  bool big_pages, bad_page;

  __device__ __forceinline__ Producer(const Params& p_, const Shared& sh_, const Item& it_, int ct)
      : p(p_), sh(sh_), it(it_) {
    lg_sub = __ffs(p.subpage) - 1;
    pool_pages = p.pool_rows >> lg_sub;
    pool = p.kv + (int64_t)it.k * p.pool_rows * kDqk * kElem;
    pages = p.page_ids + ((int64_t)it.k * p.batch + it.b) * p.max_pages;
    big_pages = p.subpage >= kTileN;  // then a tile lies inside one subpage
    bad_page = false;
    if (kFp8) {
      tk0 = ct >> 2;
      col = (ct & 3) * 16;
      soff0 = sw128_offset(tk0, 2 * (ct & 3));  // chunk 2q; chunk 2q+1 is 16 bytes away (xor)
    } else {
      tk0 = ct >> 3;
      col = (ct & 7) * 16;
      soff0 = sw128_offset(tk0, ct & 7);
    }
  }

  __device__ __forceinline__ int32_t tile_page(int i) const {
    if (!big_pages || i >= it.n_tiles) return -1;
    return __ldg(pages + ((it.t_start + i * kTileN) >> lg_sub));
  }

  // Row pointers of this thread's tokens of tile i (nullptr: masked or invalid page).
  __device__ __forceinline__ void rows(int i, int32_t pg_tile, const uint8_t* (&rp)[kToks]) {
    const int tok0 = it.t_start + i * kTileN + tk0;
#pragma unroll
    for (int j = 0; j < kToks; ++j) {
      const int li = tok0 + j * kTokStride;
      rp[j] = nullptr;
      if (li < it.t_end) {
        const int32_t pg = big_pages ? pg_tile : __ldg(pages + (li >> lg_sub));
        if (pg >= 0 && pg < pool_pages) {
          const int64_t row = ((int64_t)pg << lg_sub) + (li & (p.subpage - 1));
          rp[j] = pool + row * (kDqk * kElem) + kD0 * kElem + col;
        } else {
          bad_page = true;
        }
      }
    }
  }

  // cp.async of this thread's chunks of tile i into its staging slots (chunk l
  // at raw + l*2048 + ct*16); masked chunks are zero-filled.
  __device__ __forceinline__ void issue(int i, int32_t pg_tile, uint32_t raw) {
    const uint8_t* rp[kToks];
    rows(i, pg_tile, rp);
#pragma unroll
    for (int a = 0; a < kAtoms; ++a)
#pragma unroll
      for (int j = 0; j < kToks; ++j)
        cp_async16(raw + (a * kToks + j) * 2048, rp[j] ? rp[j] + a * 64 * kElem : pool,
                   rp[j] ? 16u : 0u);
    cp_async_commit();
  }

  // Staged tile -> registers (waits for this thread's copies).
  __device__ __forceinline__ void fetch(const uint8_t* raw, uint4 (&v)[kLoads]) {
    cp_async_wait_all();
#pragma unroll
    for (int l = 0; l < kLoads; ++l) v[l] = *reinterpret_cast<const uint4*>(raw + l * 2048);
  }

  __device__ __forceinline__ void load(int i, int32_t pg_tile, uint4 (&v)[kLoads]) {
    const uint8_t* rp[kToks];
    rows(i, pg_tile, rp);
#pragma unroll
    for (int a = 0; a < kAtoms; ++a)
#pragma unroll
      for (int j = 0; j < kToks; ++j)
        v[a * kToks + j] = rp[j] ? __ldg(reinterpret_cast<const uint4*>(rp[j] + a * 64 * kElem))
                                 : make_uint4(0u, 0u, 0u, 0u);
  }

  __device__ __forceinline__ bool store(int i, const uint4 (&v)[kLoads]) {
    const int st = i % kStages;
    if (i >= kStages && !wait_phase(&sh.bars[kBarKvEmpty + st], ((i / kStages) - 1) & 1,
                                    sh.abort_flag, p.status, false))
      return false;
    uint8_t* base = sh.stages + st * kStageBytes + soff0;
#pragma unroll
    for (int a = 0; a < kAtoms; ++a) {
#pragma unroll
      for (int j = 0; j < kToks; ++j) {
        uint8_t* dst = base + a * kAtomBytes + j * kTokStride * 128;
        const uint4 x = v[a * kToks + j];
        if (kFp8) {
          uint4 lo, hi;
          e4m3x4_to_f16x4(x.x, lo.x, lo.y);
          e4m3x4_to_f16x4(x.y, lo.z, lo.w);
          e4m3x4_to_f16x4(x.z, hi.x, hi.y);
          e4m3x4_to_f16x4(x.w, hi.z, hi.w);
          *reinterpret_cast<uint4*>(dst) = lo;
          // chunk 2q+1 = (2q ^ (tk & 7)) ^ 1 within the row: 16 bytes further or back
          *reinterpret_cast<uint4*>(reinterpret_cast<uintptr_t>(dst) ^ 16u) = hi;
        } else {
          *reinterpret_cast<uint4*>(dst) = x;
        }
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(&sh.bars[kBarKvFull + st]);
    return true;
  }

  // FP8: two tiles in flight. Registers hold tile i+1 and the shared staging
  // slots receive tile i+2 (cp.async) while this thread waits for a free stage,
  // so a freed stage is refilled by the conversion alone. BF16 (twice the bytes,
  // no room to stage): one register buffer, loaded right after the previous store.
  __device__ __forceinline__ void run(int ct) {
    const int n = it.n_tiles;
    uint4 v[kLoads];
    if (kFp8) {
      // step j: store tile j-1 (registers), fetch tile j (staging -> registers),
      // issue tile j+1 (global -> staging); one code site each
      const uint8_t* raw = sh.raw + ct * 16;
      const uint32_t raw_s = smem_u32(raw);
      for (int j = -1; j <= n; ++j) {
        const int32_t pg = tile_page(j + 1);
        if (j >= 1 && !store(j - 1, v)) break;
        if (j >= 0 && j < n) fetch(raw, v);
        if (j + 1 < n) issue(j + 1, pg, raw_s);
      }
      cp_async_wait_all();  // nothing may land in shared memory after the CTA exits
    } else {
      if (n > 0) load(0, tile_page(0), v);
      for (int i = 0; i < n; ++i) {
        const int32_t pg_next = tile_page(i + 1);
        if (!store(i, v)) break;
        if (i + 1 < n) load(i + 1, pg_next, v);
      }
    }
    if (bad_page) raise_status(p.status, DCP_STATUS_BAD_PAGE);
  }
};

// ----------------------------------------------------------------- MMA issuers
// A thread issuing tcgen05.mma back to back gets about one instruction per
// 55-130 cycles (N = 64..256), but any branch or non-trivial arithmetic between
// two of them was measured to double that. So each chain is a fully unrolled
// straight line whose descriptors are per-tile bases plus constants (the
// address field of a descriptor is the byte address / 16 in its low bits).

// The score chain: S = Q . K_tile^T over this CTA's 4*kAtoms k-steps (16 dims
// each), q from TMEM, K from the stage (K-major, 128-byte swizzle).
template <bool kFp8, int kAtoms>
__device__ __forceinline__ void run_score_chain(const Params& p, const Shared& sh, const Item& it,
                                                uint32_t tbase) {
  constexpr uint32_t idq = idesc_f16(kRows, kTileN, !kFp8, false);
  const uint32_t stage0 = smem_u32(sh.stages);
  if (wait_uniform(&sh.bars[kBarQFull], 0, sh.abort_flag, p.status, p.q_wait_ns)) {
    tc_fence_after();
    for (int i = 0; i < it.n_tiles; ++i) {
      const int st = i % kStages;
      if (!wait_uniform(&sh.bars[kBarKvFull + st], (i / kStages) & 1, sh.abort_flag, p.status))
        break;
      if (i >= 1 && !wait_uniform(&sh.bars[kBarSFree], (i - 1) & 1, sh.abort_flag, p.status))
        break;
      tc_fence_after();
      const uint64_t bdesc0 = smem_desc_sw128(stage0 + st * kStageBytes, 16, 1024);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 4 * kAtoms; ++kk)
          mma_f16_ts(tbase + kColS, tbase + kColQ + 8 * kk,
                     bdesc0 + (uint64_t)(((kk >> 2) * kAtomBytes + (kk & 3) * 32) >> 4), idq,
                     kk > 0 ? 1u : 0u);
        tc_commit(&sh.bars[kBarSFull]);
        tc_commit(&sh.bars[kBarKvEmpty + st]);
      }
      __syncwarp();
    }
  }
  // drain: every MMA issued above has completed before TMEM can be released
  tc_commit_elect(&sh.bars[kBarDrainS]);
  int never = 0;
  wait_uniform(&sh.bars[kBarDrainS], 0, &never, p.status);
}

// O += P(j) . V(j) for every tile, as soon as the softmax has written P(j).
template <bool kFp8>
__device__ __forceinline__ void run_pv(const Params& p, const Shared& sh, const Item& it,
                                       uint32_t tbase) {
  constexpr uint32_t idp = idesc_f16(kRows, 256, !kFp8, true);
  const uint32_t stage0 = smem_u32(sh.stages);
  for (int j = 0; j < it.n_tiles; ++j) {
    if (!wait_uniform(&sh.bars[kBarPFull], j & 1, sh.abort_flag, p.status)) break;
    tc_fence_after();
    const uint64_t vdesc0 = smem_desc_sw128(stage0 + (j % kStages) * kStageBytes, kAtomBytes, 1024);
    const uint32_t tp = tbase + kColP;
    const uint32_t acc0 = j > 0 ? 1u : 0u;
    if (elect_one()) {
#pragma unroll
      for (int kk = 0; kk < kTileN / 16; ++kk)
        mma_f16_ts(tbase + kColO, tp + 8 * kk, vdesc0 + (uint64_t)((kk * 2048) >> 4), idp,
                   kk > 0 ? 1u : acc0);
      tc_commit(&sh.bars[kBarODone]);
      // P.V(j) done is also an arrival on tile j+1's exchange barrier, whose waiters
      // then know the P buffer is free and O stable without a second wait
      tc_commit(&sh.bars[kBarXFull + ((j + 1) & 1)]);
      tc_commit(&sh.bars[kBarKvEmpty + (j % kStages)]);
    }
    __syncwarp();
  }
  tc_commit_elect(&sh.bars[kBarDrainP]);
  int never = 0;
  wait_uniform(&sh.bars[kBarDrainP], 0, &never, p.status);
}

// ----------------------------------------------------------------- softmax
// Rare paths live out of line so that the per-tile loop stays small in the
// instruction cache (it shares the SM with the producer and MMA warps).

// O[:, this warp's 128 columns] *= a (per-thread row factor); warp-collective.
__device__ __noinline__ void rescale_o(uint32_t tO, float a) {
  for (int c8 = 0; c8 < 8; ++c8) {
    uint32_t o[16];
    tmem_ld16(tO + 16 * c8, o);
    tmem_wait_ld16(o);
#pragma unroll
    for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
    tmem_st16(tO + 16 * c8, o);
  }
  tmem_wait_st();
}

// Stores 32 columns (c4-th group of the warp's columns) of this warp's 32 rows of the
// normalised partial output: lane r scales row r by its 1/l and writes it into a 4 KB
// shared-memory slice of this warp (chunk c of row r at 16-byte position c ^ (r mod 8)),
// then lane l stores chunk (l mod 8) of rows 4k + l/8, k = 0..7, so one instruction
// writes four whole 128-byte row segments (a store per thread of its own row would
// touch 32 rows per instruction). Rows at or past rows_left are not written.
__device__ __forceinline__ void store_o_cols(const uint32_t (&o)[32], int c4, int rows_left,
                                             float inv, float* dst0, uint4* slice) {
  const int lane = threadIdx.x & 31;
  const int rsub = lane >> 3, chunk = lane & 7;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    slice[lane * 8 + (c ^ (lane & 7))] =
        make_uint4(__float_as_uint(__uint_as_float(o[4 * c]) * inv),
                   __float_as_uint(__uint_as_float(o[4 * c + 1]) * inv),
                   __float_as_uint(__uint_as_float(o[4 * c + 2]) * inv),
                   __float_as_uint(__uint_as_float(o[4 * c + 3]) * inv));
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int row = 4 * k + rsub;
    if (row < rows_left)
      *reinterpret_cast<uint4*>(dst0 + (int64_t)row * kDv + 32 * c4 + 4 * chunk) =
          slice[row * 8 + (chunk ^ (row & 7))];
  }
  __syncwarp();  // the slice is written again for the next 32 columns
}

// This warp's 64 output columns of its 32 rows (two passes of store_o_cols). The
// second pass's tensor-memory load is in flight while the first is stored.
__device__ __noinline__ void store_o(uint32_t tO, bool have_o, int rows_left, float inv,
                                     float* dst0, uint4* slice) {
  uint32_t oa[32], ob[32];
  if (have_o) {
    tmem_ld32(tO, oa);
    tmem_ld32(tO + 32, ob);
    tmem_wait_ld(oa);
    store_o_cols(oa, 0, rows_left, inv, dst0, slice);
    tmem_wait_ld(ob);
    store_o_cols(ob, 1, rows_left, inv, dst0, slice);
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) oa[e] = 0u;
    for (int c4 = 0; c4 < 2; ++c4) store_o_cols(oa, c4, rows_left, inv, dst0, slice);
  }
}

// The packed epilogue: this warp's 32 rows of its 64 output columns, normalised and
// rounded to BF16 (nearest even), written into the all-to-all send buffer: query row
// qr of the tile is head qr mod H of verify row qr / H, whose entry lives in the chunk
// for the head's destination. 32 columns (64 bytes of a row) at a time go through the
// warp's slice: lane r writes its row's four 16-byte chunks (chunk c at position
// c ^ ((r / 2) mod 4), conflict-free), then lane l stores chunk (l mod 4) of rows
// 8k + l/4, k = 0..3, so one instruction writes eight 64-byte row segments.
// send_k: this rank's send buffer; cw: words per chunk; qr_first: the warp's first
// query row; entry_row0: verify-row index of the sequence's first row (b * qlen);
// col0: the first of the warp's output columns.
__device__ __noinline__ void store_o_packed(uint32_t tO, bool have_o, int rows_left, float inv,
                                            uint4* slice, uint16_t* send_k, int64_t cw, int H,
                                            int Hg, int qr_first, int64_t entry_row0, int col0) {
  const int lane = threadIdx.x & 31;
  const int rsub = lane >> 2, chunk = lane & 3;
  uint16_t* dst[4];  // the send-buffer entry of each row this lane stores
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int qrk = qr_first + 8 * k + rsub;
    const int jk = qrk / H, hk = qrk - jk * H;
    const int dk = hk / Hg;
    dst[k] = send_k + dk * cw + ((entry_row0 + jk) * Hg + (hk - dk * Hg)) * kDv + col0;
  }
  for (int c2 = 0; c2 < 2; ++c2) {
    uint32_t o[32];
    if (have_o) {
      tmem_ld32(tO + 32 * c2, o);
      tmem_wait_ld(o);
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = 0u;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(o[8 * c + 2 * e]) * inv,
                                                  __uint_as_float(o[8 * c + 2 * e + 1]) * inv);
        w[e] = *reinterpret_cast<uint32_t*>(&b2);
      }
      slice[lane * 4 + (c ^ ((lane >> 1) & 3))] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int row = 8 * k + rsub;
      if (row < rows_left)
        *reinterpret_cast<uint4*>(dst[k] + 32 * c2 + 8 * chunk) =
            slice[row * 4 + (chunk ^ ((row >> 1) & 3))];
    }
    __syncwarp();  // the slice is written again for the next 32 columns
  }
}

// Q slices of this warp's 32 rows into TMEM (16-bit, 2 per column; atom a at
// columns 32a); half 0 loads atoms 0-2, half 1 the rest. Reads are coalesced: for
// each atom a lane loads 16-byte chunk (lane mod 8) of row 4k + lane/8, k = 0..7, so
// one instruction covers four whole 128-byte row segments (a load per thread of its
// own row would touch 32 rows per instruction). The converted chunks go through a
// 4 KB shared-memory slice of this warp (chunk c of row r at 16-byte position
// c ^ (r mod 8), conflict-free both ways), from which lane r takes row r for the TMEM
// store. The next atom's loads are in flight while the current one is converted
// (requesting every atom at once measured slower: it raises the kernel's register
// count). Returns true if some |q| exceeds the f16 range on the FP8 path.
template <bool kFp8, int kAtoms>
__device__ __noinline__ bool load_q(const uint16_t* rows0, int rows_left, int h, uint32_t tQ,
                                    uint4* slice) {
  bool q_range = false;
  const int lane = threadIdx.x & 31;
  const int a0 = h == 0 ? 0 : 3;
  const int a1 = h == 0 ? 3 : kAtoms;
  const int rsub = lane >> 3, chunk = lane & 7;
  uint4 cur[8], nxt[8];
  auto fetch = [&](int a, uint4 (&v)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int row = 4 * k + rsub;
      v[k] = (a < a1 && row < rows_left)
                 ? __ldg(reinterpret_cast<const uint4*>(rows0 + (int64_t)row * kDqk + a * 64 +
                                                         chunk * 8))
                 : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  fetch(a0, cur);
  for (int a = a0; a < a1; ++a) {
    fetch(a + 1, nxt);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint4 x = cur[k];
      if (kFp8) {
        uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float f0 = __uint_as_float(wv[e] << 16);
          const float f1 = __uint_as_float(wv[e] & 0xFFFF0000u);
          q_range |= fabsf(f0) > 65504.f || fabsf(f1) > 65504.f;
          __half2 hh = __floats2half2_rn(f0, f1);
          wv[e] = *reinterpret_cast<uint32_t*>(&hh);
        }
        x = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      }
      const int row = 4 * k + rsub;
      slice[row * 8 + (chunk ^ (row & 7))] = x;
    }
    __syncwarp();
    uint32_t w[32];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 x = slice[lane * 8 + (c ^ (lane & 7))];
      w[4 * c] = x.x, w[4 * c + 1] = x.y, w[4 * c + 2] = x.z, w[4 * c + 3] = x.w;
    }
    __syncwarp();  // the slice is written again for the next atom
    tmem_st32(tQ + 32 * a, w);
#pragma unroll
    for (int k = 0; k < 8; ++k) cur[k] = nxt[k];
  }
  tmem_wait_st();
  return q_range;
}

// Tokens of one (row, half) whose subpage id is invalid, when subpages are
// shorter than a tile (one tile spans several subpages): clears their bits.
__device__ __noinline__ uint32_t small_page_mask(uint32_t vis, const int32_t* pages, int first_tok,
                                                 int cnt, int lg_sub, int64_t pool_pages) {
  const int first = first_tok >> lg_sub;
  const int last = (first_tok + cnt - 1) >> lg_sub;
  for (int q = first; q <= last; ++q) {
    const int32_t pg = pages[q];
    if (pg < 0 || pg >= pool_pages) {
      const int lo = max(0, (q << lg_sub) - first_tok);
      const int hi = min(32, ((q + 1) << lg_sub) - first_tok);
      const uint32_t m = (hi - lo >= 32) ? 0xFFFFFFFFu : (((1u << (hi - lo)) - 1u) << lo);
      vis &= ~m;
    }
  }
  return vis;
}

// Both 16-bit halves of a and b multiplied pairwise into f32 (exact: a product of
// two f16 values has 22 significant bits).
__device__ __forceinline__ float2 mul_f16x2_f32(uint32_t a, uint32_t b) {
  float2 r;
  asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
      "mov.b32 {a0, a1}, %2;\n\t"
      "mov.b32 {b0, b1}, %3;\n\t"
      "fma.rn.f32.f16 %0, a0, b0, 0f00000000;\n\t"
      "fma.rn.f32.f16 %1, a1, b1, 0f00000000;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "r"(a), "r"(b));
  return r;
}

// Front warps (0-7): warp w owns rows 32*(w%4) .. +31 and token half w/4 of every tile.
// Per tile: S -> own factors and half maximum -> the peer's slot and the local buffers.
// Keeps no state across tiles (the factors are relative to the half's own maximum), so
// it runs up to two tiles ahead of the back warps. Returns false on a timeout.
template <bool kFp8, int kAtoms>
__device__ __forceinline__ bool run_front(const Params& p, const Shared& sh, const Item& it,
                                          uint32_t tbase, int lane, int qw, int h, int r,
                                          int row_end, float sc) {
  constexpr int cta = kAtoms - 4;
  const uint32_t tS = tbase + ((uint32_t)(qw * 32) << 16) + kColS + 32 * h;
  const uint32_t peer = cta ^ 1;
  const uint32_t xch_remote = mapa_shared(smem_u32(sh.xch), peer);
  const uint32_t xfull_remote = mapa_shared(smem_u32(&sh.bars[kBarXFull]), peer);
  const int32_t* pages = p.page_ids + ((int64_t)it.k * p.batch + it.b) * p.max_pages;
  const int lg_sub = __ffs(p.subpage) - 1;
  const int64_t pool_pages = p.pool_rows >> lg_sub;
  const bool big_pages = p.subpage >= kTileN;
  auto wait_warp = [&](int bar, uint32_t parity, bool cluster) -> bool {
    return __all_sync(0xffffffffu,
                      wait_phase(&sh.bars[bar], parity, sh.abort_flag, p.status, cluster));
  };
  const int n = it.n_tiles;
  // own factors (f16, the words sent to the peer) by tile mod 2: [slot][half][group 4][row]
  uint4* eprev = sh.eprev + h * 4 * kRows + r;
  int32_t pg_next = (big_pages && n > 0) ? __ldg(pages + (it.t_start >> lg_sub)) : 0;
  for (int i = 0; i < n; ++i) {
    const int tok0 = it.t_start + i * kTileN;
    const int32_t pg_tile = pg_next;
    if (!wait_warp(kBarSFull, i & 1, false)) return false;
    tc_fence_after();
    float e_cur[32];
    {
      uint32_t sv[32];
      tmem_ld32(tS, sv);
      tmem_wait_ld(sv);
#pragma unroll
      for (int c = 0; c < 32; ++c) e_cur[c] = __uint_as_float(sv[c]);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.bars[kBarSFree]);
    if (big_pages && i + 1 < n) pg_next = __ldg(pages + ((tok0 + kTileN) >> lg_sub));
    // visible tokens of this row in this half: [tok0 + 32h, row_end), pages valid
    const int cnt = max(0, min(32, row_end - tok0 - 32 * h));
    const bool page_ok = !big_pages || (pg_tile >= 0 && pg_tile < pool_pages);
    // e_cur := 2^(x*sc - m*sc + 14) with x the raw partial score (sc > 0); masked
    // tokens (past the row's boundary, invalid pages) become -inf, i.e. factor 0
    uint32_t vis = cnt >= 32 ? 0xFFFFFFFFu : ((1u << cnt) - 1u);
    if (!page_ok) vis = 0;
    if (!big_pages && vis) vis = small_page_mask(vis, pages, tok0 + 32 * h, cnt, lg_sub, pool_pages);
    if (vis != 0xFFFFFFFFu) {
#pragma unroll
      for (int c = 0; c < 32; ++c) e_cur[c] = ((vis >> c) & 1u) ? e_cur[c] : -INFINITY;
    }
    float m4[4] = {e_cur[0], e_cur[1], e_cur[2], e_cur[3]};
#pragma unroll
    for (int c = 4; c < 32; ++c) m4[c & 3] = fmaxf(m4[c & 3], e_cur[c]);
    const float m_cur = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sc;  // -inf: none visible
    const float bias = m_cur == -INFINITY ? 0.f : kFactorLog2 - m_cur;
    // x*sc + bias two at a time (packed fp32 FMA), then 2^. on the MUFU unit
    const float2 sc2 = make_float2(sc, sc), bias2 = make_float2(bias, bias);
#pragma unroll
    for (int c = 0; c < 32; c += 2) {
      const float2 y = __ffma2_rn(make_float2(e_cur[c], e_cur[c + 1]), sc2, bias2);
      e_cur[c] = fast_exp2(y.x);
      e_cur[c + 1] = fast_exp2(y.y);
    }
    const int slot = i & 1;
    // slot i&1 of the local buffers is free once the back warps have finished tile i-2,
    // and the peer's slot i&1 once the peer's back warps have
    if (i >= 2 && !wait_warp(kBarEFree + slot, ((i >> 1) - 1) & 1, false)) return false;
    sh.mown[(slot * 2 + h) * kRows + r] = m_cur;
    if (i >= 2 && !wait_warp(kBarXFree + slot, ((i >> 1) - 1) & 1, true)) return false;
    // st.async: each store completes its bytes on the peer's xfull[slot], which the
    // peer armed with the slot size; no release fence is needed
    const uint32_t dst = xch_remote + slot * kXchSlotBytes;
    const uint32_t rbar = xfull_remote + 8 * slot;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint32_t w4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __half2 hh = __floats2half2_rn(e_cur[8 * g + 2 * e], e_cur[8 * g + 2 * e + 1]);
        w4[e] = *reinterpret_cast<uint32_t*>(&hh);
      }
      st_async_v4(dst + (uint32_t)(((h * 4 + g) * kRows + r) * 16), w4[0], w4[1], w4[2],
                  w4[3], rbar);
      eprev[(slot * 8 + g) * kRows] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
    st_async_b32(dst + kXchEBytes + (uint32_t)((h * kRows + r) * 4), __float_as_uint(m_cur),
                 rbar);
    // the own factors and the half maximum of tile i are in the local buffers
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.bars[kBarXFull + slot]);
  }
  return true;
}

// Back warps (8-15): warp w owns rows 32*(w%4) .. +31 and token half (w/4)%2. Per tile:
// the tile bound from both CTAs' half maxima, the lazy reference M, a rescale of O when
// M moves, P = E_own * E_peer * 2^(bound - M) into tensor memory for the P.V issuer, and
// the half's running sum l. Returns false on a timeout.
template <bool kFp8>
__device__ __forceinline__ bool run_back(const Params& p, const Shared& sh, const Item& it,
                                         uint32_t tbase, int cta, int lane, int warp, int qw,
                                         int h, int r, float& M, float& l_half) {
  const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
  const uint32_t tP = tbase + lane_off + kColP + 16 * h;
  const uint32_t tO = tbase + lane_off + kColO + 128 * h;
  const uint32_t xfree_remote = mapa_shared(smem_u32(&sh.bars[kBarXFree]), cta ^ 1);
  auto wait_warp = [&](int bar, uint32_t parity, bool cluster) -> bool {
    return __all_sync(0xffffffffu,
                      wait_phase(&sh.bars[bar], parity, sh.abort_flag, p.status, cluster));
  };
  const bool armer = warp == kFrontWarps && lane == 0;
  const uint4* eown = sh.eprev + h * 4 * kRows + r;
  const int n = it.n_tiles;
  for (int t = 0; t < n; ++t) {
    const int slot = t & 1;
    // one thread arms this use of the slot with its size (the bytes may already be in)
    if (armer) {
      mbar_arrive_expect_tx(&sh.bars[kBarXFull + slot], kXchSlotBytes);
      if (t == 0) mbar_arrive(&sh.bars[kBarXFull + slot]);  // no P.V before tile 0
    }
    // the peer's factors, the local front warps' factors and maxima, the previous P.V
    if (!wait_warp(kBarXFull + slot, (t >> 1) & 1, true)) return false;
    const uint8_t* src = sh.xch + slot * kXchSlotBytes;
    const float* mpeer = reinterpret_cast<const float*>(src + kXchEBytes);
    const float* mown = sh.mown + slot * 2 * kRows;
    // tile bound of the row: max over both halves of m_own + m_peer
    const float mo0 = mown[r], mo1 = mown[kRows + r];
    const float mp0 = mpeer[r], mp1 = mpeer[kRows + r];
    const float ub0 = (mo0 == -INFINITY || mp0 == -INFINITY) ? -INFINITY : mo0 + mp0;
    const float ub1 = (mo1 == -INFINITY || mp1 == -INFINITY) ? -INFINITY : mo1 + mp1;
    const float ub = fmaxf(ub0, ub1);
    const float ub_h = h ? ub1 : ub0;
    const bool need = ub != -INFINITY && (M == -INFINITY || ub > M + kRaiseAbove);
    float alpha = 1.f;
    if (need) {
      const float m_new = ub - kRefBelow;
      alpha = M == -INFINITY ? 0.f : fast_exp2(M - m_new);
      l_half *= alpha;
      M = m_new;
    }
    // P.V(t-1) has completed (its commit was an arrival on this tile's exchange
    // barrier): the P buffer is free and O is stable
    tc_fence_after();
    if (t >= 1 && __any_sync(0xffffffffu, need)) rescale_o(tO, need ? alpha : 1.f);
    // p = E_own * E_peer * 2^(m_own + m_peer - M); both factors carry 2^14 and are the
    // f16 words that were exchanged, so the two CTAs form bit-identical weights. 8
    // tokens per step (two steps per loop body)
    const float f = ub_h == -INFINITY ? 0.f : fast_exp2(ub_h - M - 2.0f * kFactorLog2);
    const float2 f2 = make_float2(f, f);
    float2 lsum2 = make_float2(0.f, 0.f);
    const uint4* pe_src = reinterpret_cast<const uint4*>(src) + h * 4 * kRows + r;
    const uint4* own = eown + slot * 8 * kRows;
#pragma unroll 2
    for (int g = 0; g < 4; ++g) {
      const uint4 a = own[g * kRows], b = pe_src[g * kRows];
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
      uint32_t pk[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        // two weights at a time: the exact f32 product of the two f16 factors, times f
        const float2 pp = __fmul2_rn(mul_f16x2_f32(aw[e], bw[e]), f2);
        // l sums the fp32 weights; the P.V contraction uses P rounded to 16 bits
        lsum2 = __fadd2_rn(lsum2, pp);
        if (kFp8) {
          __half2 hh = __floats2half2_rn(pp.x, pp.y);
          pk[e] = *reinterpret_cast<uint32_t*>(&hh);
        } else {
          __nv_bfloat162 hh = __floats2bfloat162_rn(pp.x, pp.y);
          pk[e] = *reinterpret_cast<uint32_t*>(&hh);
        }
      }
      tmem_st4(tP + 4 * g, pk);
    }
    __syncwarp();
    // done with the peer's slot and the local own-factor slot: the values are in
    // registers already
    if (lane == 0) {
      mbar_arrive_remote_relaxed(xfree_remote + 8 * slot);
      mbar_arrive(&sh.bars[kBarEFree + slot]);
    }
    l_half += lsum2.x + lsum2.y;
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.bars[kBarPFull]);
  }
  return true;
}

// The softmax warps: front (0-7) and back (8-15) loops, then a shared epilogue in which
// each of the 16 warps stores 64 of the CTA's 256 output columns of its 32 rows.
template <bool kFp8, int kAtoms>
__device__ __forceinline__ void run_softmax(const Params& p, const Shared& sh, const Item& it,
                                            uint32_t tbase, int tid, int warp) {
  constexpr int cta = kAtoms - 4;
  constexpr int d0 = 256 * cta;
  const int lane = tid & 31;
  const int qw = warp & 3;          // TMEM lane quarter
  const int h = (warp >> 2) & 1;    // token half of each tile / O column half
  const bool back = warp >= kFrontWarps;
  const int r = qw * 32 + lane;
  const int qrows = p.qlen * p.H;
  const int R = p.batch * p.qlen;
  const bool row_ok = r < it.rows_valid;
  const int qr = it.qr0 + r;
  const int j = row_ok ? qr / p.H : 0;
  const float kv_scale = p.kv_scale ? *p.kv_scale : 1.0f;
  const int n = it.n_tiles;
  auto wait_warp = [&](int bar, uint32_t parity, bool cluster) -> bool {
    return __all_sync(0xffffffffu,
                      wait_phase(&sh.bars[bar], parity, sh.abort_flag, p.status, cluster));
  };

  float M = -INFINITY;  // running reference (log2 units), same in both CTAs (back warps)
  float l_half = 0.f;   // sum of this half's weights (back warps)
  bool ok;
  if (!back) {
    {
      // this warp's 32 rows start at row qw*32 of the tile; the own-factor buffer, first
      // written after the first scores (which need every warp's q), lends each warp a
      // 4 KB slice for the transpose
      const int r_first = qw * 32;
      const uint16_t* rows0 = p.q + ((int64_t)it.b * qrows + it.qr0 + r_first) * kDqk + d0;
      const uint32_t tQ = tbase + ((uint32_t)(qw * 32) << 16) + kColQ;
      const bool q_range = load_q<kFp8, kAtoms>(rows0, it.rows_valid - r_first, h, tQ,
                                                sh.eprev + warp * 256);
      tc_fence_before();
      if (q_range) raise_status(p.status, DCP_STATUS_Q_RANGE);
      __syncwarp();
      if (lane == 0 && !p.hold_q) mbar_arrive(&sh.bars[kBarQFull]);
    }
    cluster_wait();  // the peer's barriers are initialised before this warp's first send
    const int L = row_ok ? p.row_len[(int64_t)it.k * R + (int64_t)it.b * p.qlen + j] : 0;
    const int row_end = min(L, it.t_end);  // tokens at or past it are invisible to this row
    const float sc = p.softmax_scale * kv_scale * kLog2e;
    ok = run_front<kFp8, kAtoms>(p, sh, it, tbase, lane, qw, h, r, row_end, sc);
  } else {
    ok = run_back<kFp8>(p, sh, it, tbase, cta, lane, warp, qw, h, r, M, l_half);
  }

  // epilogue: the back warps combine both halves' l into the row's output scale; every
  // softmax warp then stores 64 O columns of its rows
  const bool have_o =
      __all_sync(0xffffffffu, ok) && n > 0 && wait_warp(kBarODone, (n - 1) & 1, false);
  tc_fence_after();
  float inv = 0.f, l_run = 0.f;
  if (back) {
    sh.lcomb[h * kRows + r] = l_half;
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.bars[kBarLComb]);
    const bool paired = wait_warp(kBarLComb, 0, false);
    l_run = l_half + sh.lcomb[(h ^ 1) * kRows + r];
    inv = (paired && l_run > 0.f) ? kv_scale / l_run : 0.f;
    if (h == 0) sh.einv[r] = inv;
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.bars[kBarEpi]);
  } else if (wait_warp(kBarEpi, 0, false)) {
    inv = sh.einv[r];
  }
  const int col_w = 128 * h + (back ? 64 : 0);  // the warp's columns within the CTA's 256
  const uint32_t tO = tbase + ((uint32_t)(qw * 32) << 16) + kColO + col_w;
  const int64_t rh = (int64_t)it.b * qrows + qr;
  const int64_t base = ((int64_t)it.k * p.num_splits + it.s) * ((int64_t)R * p.H) + rh;
  // every MMA has completed (or none ran), so the KV stages are free and lend each warp
  // a 4 KB slice for the transpose
  uint4* slice = reinterpret_cast<uint4*>(sh.stages) + warp * 256;
  const bool lse_owner = back && row_ok && cta == 0 && h == 0;
  if (p.send != nullptr) {
    // packed epilogue
    const int Hg = p.H / p.G;
    store_o_packed(tO, have_o, it.rows_valid - qw * 32, inv, slice,
                   p.send + (int64_t)it.k * p.G * p.send_cw, p.send_cw, p.H, Hg,
                   it.qr0 + qw * 32, (int64_t)it.b * p.qlen, 256 * cta + col_w);
    if (lse_owner) {
      // the LSE words (low 16 bits, then high), as one 32-bit store
      const float lse = l_run > 0.f ? (M + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
      const int hh = qr - j * p.H, dd = hh / Hg;
      const int64_t entry = ((int64_t)it.b * p.qlen + j) * Hg + (hh - dd * Hg);
      uint16_t* cbase = p.send + ((int64_t)it.k * p.G + dd) * p.send_cw;
      *reinterpret_cast<uint32_t*>(cbase + (int64_t)R * Hg * kDv + entry * 2) =
          __float_as_uint(lse);
    }
    if (cta == 0 && it.b == 0 && it.t == 0 && tid == 0) {
      // the zero words that end each of this rank's chunks
      const int64_t used = (int64_t)R * Hg * (kDv + 2);
      for (int dd = 0; dd < p.G; ++dd)
        for (int64_t w = used; w < p.send_cw; ++w)
          p.send[((int64_t)it.k * p.G + dd) * p.send_cw + w] = 0;
    }
    return;
  }
  const int64_t base0 = base - r + qw * 32;
  store_o(tO, have_o, it.rows_valid - qw * 32, inv,
          p.part_o + base0 * kDv + 256 * cta + col_w, slice);
  if (lse_owner) {
    p.part_m[base] = l_run > 0.f ? M : -INFINITY;
    p.part_l[base] = l_run;
    if (it.s == 0) {
      // the empty slots s >= 1 of this (rank, sequence) run no item of their own when
      // the order kernel drops them: their m and l are written here (their output
      // is never read)
      const int64_t sb0 = ((int64_t)it.k * p.batch + it.b) * p.num_splits;
      const int64_t slot = (int64_t)R * p.H;
      for (int s2 = 1; s2 < p.num_splits; ++s2) {
        if (p.split_end[sb0 + s2] <= p.split_beg[sb0 + s2]) {
          p.part_m[base + s2 * slot] = -INFINITY;
          p.part_l[base + s2 * slot] = 0.f;
        }
      }
    }
  }
}

// ----------------------------------------------------------------- schedule
// The hardware hands clusters out in index order as SMs free up, so items whose
// tile counts differ widely (sequences of very different lengths) finish unevenly.
// order_kernel sorts the items by tile count, longest first, which brings list
// scheduling within a few percent of the ideal makespan. The sort is over groups
// (rank, sequence, split): a group's row tiles read the same cache rows, so they
// stay adjacent and run side by side, sharing those rows in L2. Groups of empty
// slots s >= 1 (split_beg == split_end) are left out; slot 0's items write their
// m and l. One CTA: a histogram over (clamped) group tile counts, an exclusive
// scan, a scatter; then the number of listed items. Groups with equal counts land
// in any order; no item's result depends on the cluster that computes it.
constexpr int kOrderThreads = 1024;
constexpr int kOrderBuckets = 4096;  // tile counts at or above the last bucket share it
constexpr int kOrderMaxItems = 1 << 16;

__global__ void __launch_bounds__(kOrderThreads) order_kernel(const Params p, int n_groups,
                                                              int32_t* order) {
  __shared__ int bucket[kOrderBuckets];
  __shared__ int warp_total[kOrderThreads / 32];
  const int tid = threadIdx.x;
  for (int b = tid; b < kOrderBuckets; b += kOrderThreads) bucket[b] = 0;
  __syncthreads();
  const int rt = p.n_row_tiles;
  // group g = (rank, sequence, split) in natural order is also its split-bound index
  auto dropped = [&](int g) {
    return g % p.num_splits != 0 && p.split_end[g] <= p.split_beg[g];
  };
  auto key_of = [&](int g) {
    int tiles = 0;
    for (int t = 0; t < rt; ++t) tiles = max(tiles, decode_item(p, g * rt + t).n_tiles);
    return kOrderBuckets - 1 - min(tiles, kOrderBuckets - 1);
  };
  for (int g = tid; g < n_groups; g += kOrderThreads)
    if (!dropped(g)) atomicAdd(&bucket[key_of(g)], 1);
  __syncthreads();
  // exclusive scan of the buckets, 4 per thread
  constexpr int kPer = kOrderBuckets / kOrderThreads;
  int cnt[kPer], sum = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    cnt[j] = bucket[tid * kPer + j];
    sum += cnt[j];
  }
  const int lane = tid & 31, wid = tid >> 5;
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_total[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int t = warp_total[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += v;
    }
    warp_total[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  int excl = incl - sum + (wid > 0 ? warp_total[wid - 1] : 0);
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    bucket[tid * kPer + j] = excl;
    excl += cnt[j];
  }
  __syncthreads();
  for (int g = tid; g < n_groups; g += kOrderThreads) {
    if (dropped(g)) continue;
    const int pos = atomicAdd(&bucket[key_of(g)], 1);
    for (int t = 0; t < rt; ++t) order[pos * rt + t] = g * rt + t;
  }
  // listed groups = the inclusive total over all warps
  if (tid == 0) order[n_groups * rt] = warp_total[kOrderThreads / 32 - 1] * rt;
}

template <bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    partial_tc_kernel(const Params p) {
  extern __shared__ unsigned char smem_raw[];
  const Shared sh = carve(smem_raw);
  const int tid = threadIdx.x;
  // warp-uniform by construction (the shuffle tells the compiler so): TMEM and
  // tcgen05 operands derived from it need no per-lane serialisation
  const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
  const int cta = (int)cluster_ctarank();
  const int cluster_id = blockIdx.x >> 1;
  // the listed count and this cluster's entry are read together (the entry is in
  // bounds either way); clusters past the listed items have nothing to do (both CTAs
  // of a cluster agree, and neither has touched a barrier or tensor memory yet)
  const int n_live = p.n_live != nullptr ? *p.n_live : INT_MAX;
  const int item = p.item_order != nullptr ? p.item_order[cluster_id] : cluster_id;
  if (cluster_id >= n_live) return;

  // barriers and tensor memory while the item's metadata loads are in flight
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sh.bars[kBarKvFull + i], 128);
      mbar_init(&sh.bars[kBarKvEmpty + i], 2);
    }
    mbar_init(&sh.bars[kBarSFull], 1);
    mbar_init(&sh.bars[kBarSFree], kFrontWarps);
    mbar_init(&sh.bars[kBarPFull], kBackWarps);
    mbar_init(&sh.bars[kBarODone], 1);
    mbar_init(&sh.bars[kBarQFull], kFrontWarps);
    for (int i = 0; i < kXchSlots; ++i) {
      // armed by one back-warp thread with the slot's bytes; the 8 front warps arrive,
      // and the completion of the previous tile's P.V (tile 0: the arming thread again)
      mbar_init(&sh.bars[kBarXFull + i], 2 + kFrontWarps);
      mbar_init(&sh.bars[kBarXFree + i], kBackWarps);
      mbar_init(&sh.bars[kBarEFree + i], kBackWarps);
    }
    mbar_init(&sh.bars[kBarLComb], kBackWarps);
    mbar_init(&sh.bars[kBarEpi], kBackWarps);
    mbar_init(&sh.bars[kBarDrainS], 1);
    mbar_init(&sh.bars[kBarDrainP], 1);
    *sh.abort_flag = 0;
    fence_mbarrier_init_cluster();
  }
  if (warp == kMmaWarpS) {
    tmem_alloc(sh.tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  const Item it = decode_item(p, item);
  if (tid == 0 && cta == 0 && it.t == 0 && it.bad_split) raise_status(p.status, DCP_STATUS_BAD_SPLIT);
  tc_fence_before();
  __syncthreads();
  // this CTA's barriers are ready for the peer. A thread waits for the peer's only where
  // it first needs them: the front warps before their first send (their q load runs
  // meanwhile), every other warp here
  cluster_arrive();
  if (warp >= kFrontWarps) cluster_wait();
  tc_fence_after();
  const uint32_t tbase = __shfl_sync(0xffffffffu, *sh.tmem_slot, 0);

  if (warp < kSoftWarps) {
    if (cta == 0) run_softmax<kFp8, 4>(p, sh, it, tbase, tid, warp);
    else run_softmax<kFp8, 5>(p, sh, it, tbase, tid, warp);
  } else if (warp < kMmaWarpS) {
    const int ct = tid - kProdWarp0 * 32;
    if (cta == 0) Producer<kFp8, 4>(p, sh, it, ct).run(ct);
    else Producer<kFp8, 5>(p, sh, it, ct).run(ct);
  } else if (warp == kMmaWarpS) {
    if (cta == 0) run_score_chain<kFp8, 4>(p, sh, it, tbase);
    else run_score_chain<kFp8, 5>(p, sh, it, tbase);
  } else if (warp == kMmaWarpP) {
    run_pv<kFp8>(p, sh, it, tbase);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer no longer touches this CTA's shared memory
  if (warp == kMmaWarpS) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_partial(const dcp_mla_dims& d, const Derived& x, const void* q,
                           const void* kv, dcp_kv_dtype kv_dtype, const float* kv_scale,
                           float softmax_scale, int num_ranks, const int32_t* row_len,
                           const int32_t* page_ids, const int32_t* split_beg,
                           const int32_t* split_end, float* part_o, float* part_m,
                           float* part_l, void* workspace, uint32_t* status,
                           cudaStream_t stream, void* send, uint64_t hold_q_ns) {
  Params p;
  p.q = reinterpret_cast<const uint16_t*>(q);
  p.kv = reinterpret_cast<const uint8_t*>(kv);
  p.kv_scale = kv_scale;
  p.row_len = row_len;
  p.page_ids = page_ids;
  p.split_beg = split_beg;
  p.split_end = split_end;
  p.part_o = part_o;
  p.part_m = part_m;
  p.part_l = part_l;
  p.status = status;
  p.item_order = nullptr;
  p.n_live = nullptr;
  p.hold_q = hold_q_ns > 0 ? 1 : 0;
  p.q_wait_ns = hold_q_ns > 0 ? hold_q_ns : kTimeoutNs;
  p.send = reinterpret_cast<uint16_t*>(send);
  p.G = d.dcp;
  p.send_cw = send ? a2a_chunk_words(d.batch * d.qlen, d.num_heads / d.dcp, kDv) : 0;
  p.softmax_scale = softmax_scale;
  p.batch = d.batch;
  p.qlen = d.qlen;
  p.H = d.num_heads;
  p.num_splits = d.num_splits;
  p.subpage = x.subpage;
  p.max_pages = x.max_pages;
  p.n_row_tiles = (d.qlen * d.num_heads + kRows - 1) / kRows;
  p.pool_rows = (int64_t)d.num_blocks * d.block_size;
  const int64_t items = (int64_t)p.n_row_tiles * d.num_splits * d.batch * num_ranks;
  if (items * 2 > INT32_MAX) return cudaErrorInvalidConfiguration;
  const bool fp8 = kv_dtype == DCP_KV_FP8_E4M3;
  auto kern = fp8 ? partial_tc_kernel<true> : partial_tc_kernel<false>;
  static bool attr_set[2][64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[fp8][dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[fp8][dev] = true;
  }
  if (workspace != nullptr && items <= kOrderMaxItems) {
    int32_t* order = reinterpret_cast<int32_t*>(workspace);
    order_kernel<<<1, kOrderThreads, 0, stream>>>(p, (int)(items / p.n_row_tiles), order);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    p.item_order = order;
    p.n_live = order + items;
  }
  kern<<<(unsigned)(items * 2), kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

size_t partial_workspace_bytes(const dcp_mla_dims& d, int num_ranks) {
  const int64_t items = (int64_t)((d.qlen * d.num_heads + kRows - 1) / kRows) * d.num_splits *
                        d.batch * num_ranks;
  return (size_t)(((items + 1) * 4 + 15) / 16 * 16);  // the order, then the listed count
}

int partial_concurrent_items() {
  static int cached[64] = {};
  int dev = 0;
  const cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess || dev < 0 || dev >= 64) {
    fail(DCP_ERR_CUDA, "no usable CUDA device: %s",
         de != cudaSuccess ? cudaGetErrorString(de) : "device index out of range");
    return -1;
  }
  if (cached[dev] > 0) return cached[dev];
  // both instantiations take the same threads and shared memory
  auto kern = partial_tc_kernel<true>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) {
    fail(DCP_ERR_CUDA, "partial kernel shared-memory attribute: %s", cudaGetErrorString(e));
    return -1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 4096);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;  // cluster shape from the kernel's own attribute
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
  if (e != cudaSuccess || n < 1) {
    cudaFuncAttributes fa = {};
    cudaFuncGetAttributes(&fa, kern);
    fail(DCP_ERR_CUDA,
         "partial kernel occupancy: %s, %d clusters (%d threads of %d registers, at most %d "
         "threads per block; %zu bytes of shared memory)",
         cudaGetErrorString(e), n, kThreads, fa.numRegs, fa.maxThreadsPerBlock, kSmemBytes);
    return -1;
  }
  cached[dev] = n;
  return n;
}

}  // namespace dcpmla
