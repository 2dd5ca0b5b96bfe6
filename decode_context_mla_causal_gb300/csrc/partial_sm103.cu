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
//   * Both CTAs need the full scores S = Q.K^T. Instead of computing them twice,
//     the 576 q/k dims are split too: CTA0 computes the partial S over dims
//     [0, 256), CTA1 over dims [256, 576); each writes its partial into the other
//     CTA's shared memory (distributed shared memory) and adds the one it gets.
//     Float addition commutes, so both CTAs hold bit-identical S, run the same
//     online softmax and agree on P, m and l.
//   * CTA c stages the dims [256c, 256c + 256 + 64c) of every token: its QK
//     slice, which also contains its value slice.
//
// Per CTA (288 threads):
//   warps 0-3  softmax: thread r owns tile row r (TMEM lane r); loads Q into
//              TMEM, exchanges partial scores, online base-2 softmax with lazy
//              rescaling, writes P (16-bit) into TMEM, final epilogue.
//   warps 4-7  KV producers: 16-byte loads of the paged cache rows (subpage ids
//              from the metadata, bounds-checked), FP8 E4M3 -> f16 conversion,
//              stores into 128-byte-swizzled K-major tiles of a 4-stage ring.
//   warp 8     TMEM allocation and the single MMA-issuing thread:
//              S  = Q[tmem] . K_tile^T        (M=128, N=64,  K=16 per MMA)
//              O += P[tmem] . V_tile          (M=128, N=256, V read MN-major
//                                              from the same swizzled tile)
// TMEM columns: O [0,256), S [256,320), P [320,352), Q [352, 352 + 32*atoms).
// The FP8-cache path computes in f16 (E4M3 -> f16 is exact; q is BF16 -> f16,
// exact in f16's normal range; |q| > 65504 sets DCP_STATUS_Q_RANGE); the BF16
// cache path computes in bf16. Accumulation is fp32 throughout.
//
// Every wait is bounded (DCP_STATUS_TIMEOUT and an orderly exit: all roles stop,
// in-flight MMAs are drained, TMEM is freed). Nothing traps.
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
constexpr int kStages = 4;     // KV ring depth
constexpr int kMaxAtoms = 5;   // 64-dim swizzle atoms staged per CTA (CTA1: 320 dims)
constexpr int kAtomBytes = kTileN * 128;
constexpr int kStageBytes = kMaxAtoms * kAtomBytes;
constexpr int kXchBytes = kTileN * kRows * 4;
constexpr int kThreads = 288;
constexpr uint32_t kColO = 0, kColS = 256, kColP = 320, kColQ = 352;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // P may grow to 2^8 before O is rescaled
constexpr uint64_t kTimeoutNs = 4000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

// barrier slots
enum {
  kBarKvFull = 0,
  kBarKvEmpty = kBarKvFull + kStages,
  kBarSFull = kBarKvEmpty + kStages,
  kBarSFree,
  kBarPFull,
  kBarODone,
  kBarQFull,
  kBarXFull,   // the peer's partial scores are in my exchange buffer
  kBarXFree,   // the peer has consumed what I wrote into its buffer
  kBarDrain,
  kNumBars
};

constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + kStages * kStageBytes + kXchBytes +
                              kNumBars * 8 + 16;

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
  float softmax_scale;
  int batch, qlen, H, num_splits, subpage, max_pages, n_row_tiles;
  int64_t pool_rows;  // rows of one rank's pool: num_blocks * block_size
};

struct Shared {
  uint8_t* stages;
  float* xbuf;
  uint64_t* bars;
  uint32_t* tmem_slot;
  int* abort_flag;
};

__device__ __forceinline__ Shared carve(unsigned char* raw) {
  Shared s;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  s.stages = base;
  s.xbuf = reinterpret_cast<float*>(base + kStages * kStageBytes);
  s.bars = reinterpret_cast<uint64_t*>(base + kStages * kStageBytes + kXchBytes);
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.bars + kNumBars);
  s.abort_flag = reinterpret_cast<int*>(s.tmem_slot + 1);
  return s;
}

// Bounded wait on an mbarrier phase. Returns false (after raising the abort flag
// and DCP_STATUS_TIMEOUT) if the phase does not complete within kTimeoutNs, or
// at once if another thread of the CTA has already aborted.
__device__ __noinline__ bool wait_phase(uint64_t* bar, uint32_t parity, int* abort_flag,
                                        uint32_t* status, bool cluster_acquire) {
  const uint32_t a = smem_u32(bar);
  if (cluster_acquire ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (cluster_acquire ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity)) return true;
    if ((it & 63u) == 0) {
      if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
      if (globaltimer_ns() - t0 > kTimeoutNs) {
        *reinterpret_cast<volatile int*>(abort_flag) = 1;
        raise_status(status, DCP_STATUS_TIMEOUT);
        return false;
      }
    }
  }
}

struct Item {
  int k, b, s, t;
  int qr0, rows_valid;
  int t_start, t_end, n_tiles;
};

__device__ __forceinline__ Item decode_item(const Params& p, int cluster_id) {
  Item it;
  int rest = cluster_id;
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
  if (beg < 0 || end < beg || end > p.max_pages) beg = end = 0;  // status raised once below
  it.t_start = beg * p.subpage;
  it.t_end = min(end * p.subpage, maxL);
  it.n_tiles = it.t_end > it.t_start ? (it.t_end - it.t_start + kTileN - 1) / kTileN : 0;
  return it;
}

// E4M3 x2 -> f16 x2 (exact): the hardware conversion.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_bytes & 0xFFFFu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// ----------------------------------------------------------------- producers
template <bool kFp8>
__device__ __forceinline__ void run_producer(const Params& p, const Shared& sh, const Item& it,
                                             int cta, int ct) {
  constexpr int kElem = kFp8 ? 1 : 2;
  const int n_atoms = 4 + cta;
  const int d0 = 256 * cta;
  // 16-byte pieces per token: FP8 -> 4 per atom (16 dims), BF16 -> 8 per atom (8 dims)
  const int ppt = n_atoms * (kFp8 ? 4 : 8);
  const int pieces = kTileN * ppt;
  constexpr int kMaxLoads = kFp8 ? (kTileN * kMaxAtoms * 4) / 128 : (kTileN * kMaxAtoms * 8) / 128;
  const int R = p.batch * p.qlen;
  (void)R;
  const int64_t pool_pages = p.pool_rows / p.subpage;
  const uint8_t* pool = p.kv + (int64_t)it.k * p.pool_rows * kDqk * kElem;
  const int32_t* pages = p.page_ids + ((int64_t)it.k * p.batch + it.b) * p.max_pages;
  bool bad_page = false;
  for (int i = 0; i < it.n_tiles; ++i) {
    const int st = i % kStages;
    const int tok0 = it.t_start + i * kTileN;
    uint4 v[kMaxLoads];
#pragma unroll
    for (int l = 0; l < kMaxLoads; ++l) {
      const int f = l * 128 + ct;
      v[l] = make_uint4(0u, 0u, 0u, 0u);
      if (f < pieces) {
        const int tk = f / ppt, pc = f % ppt;
        const int li = tok0 + tk;
        if (li < it.t_end) {
          const int32_t pg = pages[li / p.subpage];
          if (pg >= 0 && pg < pool_pages) {
            const uint8_t* src = pool + (((int64_t)pg * p.subpage + li % p.subpage) * kDqk + d0) * kElem +
                                 pc * 16;
            v[l] = __ldg(reinterpret_cast<const uint4*>(src));
          } else {
            bad_page = true;
          }
        }
      }
    }
    if (i >= kStages) {
      if (!wait_phase(&sh.bars[kBarKvEmpty + st], ((i / kStages) - 1) & 1, sh.abort_flag, p.status,
                      false))
        break;
    }
    uint8_t* stage = sh.stages + st * kStageBytes;
#pragma unroll
    for (int l = 0; l < kMaxLoads; ++l) {
      const int f = l * 128 + ct;
      if (f < pieces) {
        const int tk = f / ppt, pc = f % ppt;
        if (kFp8) {
          const int atom = pc >> 2, ch = (pc & 3) * 2;
          uint4 lo, hi;
          lo.x = e4m3x2_to_f16x2(v[l].x);
          lo.y = e4m3x2_to_f16x2(v[l].x >> 16);
          lo.z = e4m3x2_to_f16x2(v[l].y);
          lo.w = e4m3x2_to_f16x2(v[l].y >> 16);
          hi.x = e4m3x2_to_f16x2(v[l].z);
          hi.y = e4m3x2_to_f16x2(v[l].z >> 16);
          hi.z = e4m3x2_to_f16x2(v[l].w);
          hi.w = e4m3x2_to_f16x2(v[l].w >> 16);
          uint8_t* a = stage + atom * kAtomBytes;
          *reinterpret_cast<uint4*>(a + sw128_offset(tk, ch)) = lo;
          *reinterpret_cast<uint4*>(a + sw128_offset(tk, ch + 1)) = hi;
        } else {
          const int atom = pc >> 3, ch = pc & 7;
          *reinterpret_cast<uint4*>(stage + atom * kAtomBytes + sw128_offset(tk, ch)) = v[l];
        }
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(&sh.bars[kBarKvFull + st]);
  }
  if (bad_page) raise_status(p.status, DCP_STATUS_BAD_PAGE);
}

// ----------------------------------------------------------------- MMA issuer
template <bool kFp8>
__device__ __forceinline__ void run_mma(const Params& p, const Shared& sh, const Item& it, int cta,
                                        uint32_t tbase) {
  const int n_atoms = 4 + cta;
  const uint32_t idq = idesc_f16(kRows, kTileN, !kFp8, false);
  const uint32_t idp = idesc_f16(kRows, 256, !kFp8, true);
  const uint32_t stage0 = smem_u32(sh.stages);
  bool ok = wait_phase(&sh.bars[kBarQFull], 0, sh.abort_flag, p.status, false);
  tc_fence_after();
  auto issue_pv = [&](int j) -> bool {
    if (!wait_phase(&sh.bars[kBarPFull], j & 1, sh.abort_flag, p.status, false)) return false;
    tc_fence_after();
    const uint32_t sa = stage0 + (j % kStages) * kStageBytes;
#pragma unroll
    for (int kk = 0; kk < kTileN / 16; ++kk) {
      const uint64_t d = smem_desc_sw128(sa + kk * 2048, kAtomBytes, 1024);
      mma_f16_ts(tbase + kColO, tbase + kColP + 8 * kk, d, idp, (j > 0 || kk > 0) ? 1u : 0u);
    }
    tc_commit(&sh.bars[kBarODone]);
    tc_commit(&sh.bars[kBarKvEmpty + (j % kStages)]);
    return true;
  };
  for (int i = 0; ok && i < it.n_tiles; ++i) {
    const int st = i % kStages;
    if (!wait_phase(&sh.bars[kBarKvFull + st], (i / kStages) & 1, sh.abort_flag, p.status, false))
      break;
    if (i >= 1 && !wait_phase(&sh.bars[kBarSFree], (i - 1) & 1, sh.abort_flag, p.status, false))
      break;
    tc_fence_after();
    const uint32_t sa = stage0 + st * kStageBytes;
    for (int kk = 0; kk < n_atoms * 4; ++kk) {
      const uint64_t d = smem_desc_sw128(sa + (kk >> 2) * kAtomBytes + (kk & 3) * 32, 16, 1024);
      mma_f16_ts(tbase + kColS, tbase + kColQ + 8 * kk, d, idq, kk > 0 ? 1u : 0u);
    }
    tc_commit(&sh.bars[kBarSFull]);
    if (i >= 1 && !issue_pv(i - 1)) {
      ok = false;
      break;
    }
  }
  if (ok && it.n_tiles > 0 && !*reinterpret_cast<volatile int*>(sh.abort_flag))
    issue_pv(it.n_tiles - 1);
  // drain: every MMA issued above has completed before TMEM can be released
  tc_commit(&sh.bars[kBarDrain]);
  int* dummy_abort = sh.abort_flag;
  int never = 0;
  wait_phase(&sh.bars[kBarDrain], 0, &never, p.status, false);
  (void)dummy_abort;
}

// ----------------------------------------------------------------- softmax
template <bool kFp8>
__device__ __forceinline__ void run_softmax(const Params& p, const Shared& sh, const Item& it,
                                            int cta, uint32_t tbase, int r) {
  const int warp = r >> 5;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  const uint32_t tS = tbase + lane_off + kColS;
  const uint32_t tP = tbase + lane_off + kColP;
  const uint32_t tO = tbase + lane_off + kColO;
  const uint32_t tQ = tbase + lane_off + kColQ;
  const int n_atoms = 4 + cta;
  const int d0 = 256 * cta;
  const int qrows = p.qlen * p.H;
  const int R = p.batch * p.qlen;
  const bool row_ok = r < it.rows_valid;
  const int qr = it.qr0 + r;
  const int j = row_ok ? qr / p.H : 0;
  const int L = row_ok ? p.row_len[(int64_t)it.k * R + (int64_t)it.b * p.qlen + j] : 0;
  const float kv_scale = p.kv_scale ? *p.kv_scale : 1.0f;
  const float sc = p.softmax_scale * kv_scale * kLog2e;

  // Q slice -> TMEM (16-bit pairs along the dims, lane = row)
  {
    const uint16_t* src = p.q + ((int64_t)it.b * qrows + qr) * kDqk + d0;
    bool q_range = false;
    for (int a = 0; a < n_atoms; ++a) {
      uint32_t w[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row_ok) v = __ldg(reinterpret_cast<const uint4*>(src + a * 64 + c * 8));
        uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (kFp8) {
            const float f0 = __uint_as_float(x[e] << 16);
            const float f1 = __uint_as_float(x[e] & 0xFFFF0000u);
            q_range |= fabsf(f0) > 65504.f || fabsf(f1) > 65504.f;
            __half2 h = __floats2half2_rn(f0, f1);
            w[c * 4 + e] = *reinterpret_cast<uint32_t*>(&h);
          } else {
            w[c * 4 + e] = x[e];
          }
        }
      }
      tmem_st32(tQ + 32 * a, w);
    }
    tmem_wait_st();
    if (q_range) raise_status(p.status, DCP_STATUS_Q_RANGE);
    tc_fence_before();
    mbar_arrive(&sh.bars[kBarQFull]);
  }

  const int peer = cta ^ 1;
  const uint32_t x_local = smem_u32(sh.xbuf);
  const uint32_t x_remote = mapa_shared(x_local, peer);
  const uint32_t xfull_remote = mapa_shared(smem_u32(&sh.bars[kBarXFull]), peer);
  const uint32_t xfree_remote = mapa_shared(smem_u32(&sh.bars[kBarXFree]), peer);
  const int32_t* pages = p.page_ids + ((int64_t)it.k * p.batch + it.b) * p.max_pages;
  const int64_t pool_pages = p.pool_rows / p.subpage;

  // Waits are made warp-uniform: the tcgen05.ld/st that follow are warp-collective.
  auto wait_warp = [&](int bar, uint32_t parity, bool cluster) -> bool {
    return __all_sync(0xffffffffu, wait_phase(&sh.bars[bar], parity, sh.abort_flag, p.status, cluster));
  };
  float m_run = -INFINITY, l_run = 0.f;
  bool ok = true;
  for (int i = 0; i < it.n_tiles; ++i) {
    if (!wait_warp(kBarSFull, i & 1, false)) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t s0[32], s1[32];
    tmem_ld32(tS, s0);
    tmem_ld32(tS + 32, s1);
    tmem_wait_ld(s0);
    tmem_wait_ld(s1);
    tc_fence_before();
    mbar_arrive(&sh.bars[kBarSFree]);

    // exchange partial scores with the peer CTA
    if (i >= 1 && !wait_warp(kBarXFree, (i - 1) & 1, true)) {
      ok = false;
      break;
    }
#pragma unroll
    for (int g = 0; g < 8; ++g)
      st_cluster_v4(x_remote + (uint32_t)((g * kRows + r) * 16), s0[4 * g], s0[4 * g + 1],
                    s0[4 * g + 2], s0[4 * g + 3]);
#pragma unroll
    for (int g = 0; g < 8; ++g)
      st_cluster_v4(x_remote + (uint32_t)(((8 + g) * kRows + r) * 16), s1[4 * g], s1[4 * g + 1],
                    s1[4 * g + 2], s1[4 * g + 3]);
    mbar_arrive_remote(xfull_remote);
    if (!wait_warp(kBarXFull, i & 1, true)) {
      ok = false;
      break;
    }
    float sv[64];
#pragma unroll
    for (int g = 0; g < 16; ++g) {
      const float4 o = *reinterpret_cast<const float4*>(sh.xbuf + (g * kRows + r) * 4);
      const uint32_t* mine = g < 8 ? &s0[4 * g] : &s1[4 * (g - 8)];
      sv[4 * g + 0] = __uint_as_float(mine[0]) + o.x;
      sv[4 * g + 1] = __uint_as_float(mine[1]) + o.y;
      sv[4 * g + 2] = __uint_as_float(mine[2]) + o.z;
      sv[4 * g + 3] = __uint_as_float(mine[3]) + o.w;
    }
    mbar_arrive_remote(xfree_remote);

    // which of the 64 tokens are visible to this row
    const int tok0 = it.t_start + i * kTileN;
    uint64_t vis;
    {
      const int cnt_split = min(kTileN, it.t_end - tok0);
      const int cnt_row = max(0, min(cnt_split, L - tok0));
      vis = cnt_row >= 64 ? ~0ull : ((1ull << cnt_row) - 1ull);
      if (p.subpage >= kTileN) {
        const int32_t pg = pages[tok0 / p.subpage];
        if (pg < 0 || pg >= pool_pages) vis = 0;
      } else {
        const int np = (cnt_split + p.subpage - 1) / p.subpage;
        for (int q = 0; q < np; ++q) {
          const int32_t pg = pages[tok0 / p.subpage + q];
          if (pg < 0 || pg >= pool_pages) {
            const uint64_t m = (p.subpage >= 64 ? ~0ull : ((1ull << p.subpage) - 1ull))
                               << (q * p.subpage);
            vis &= ~m;
          }
        }
      }
    }
    float m_tile = -INFINITY;
#pragma unroll
    for (int c = 0; c < 64; ++c) {
      sv[c] *= sc;
      if ((vis >> c) & 1ull) m_tile = fmaxf(m_tile, sv[c]);
    }
    const float m_new = fmaxf(m_run, m_tile);
    const bool need = m_new > m_run + kRescaleThreshold || (m_run == -INFINITY && m_new != -INFINITY);
    float alpha = 1.f;
    if (need) {
      alpha = m_run == -INFINITY ? 0.f : exp2f(m_run - m_new);
      l_run *= alpha;
      m_run = m_new;
    }
    uint32_t pk[32];
    float lsum = 0.f;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const bool v0 = (vis >> (2 * c)) & 1ull, v1 = (vis >> (2 * c + 1)) & 1ull;
      const float p0 = v0 ? exp2f(sv[2 * c] - m_run) : 0.f;
      const float p1 = v1 ? exp2f(sv[2 * c + 1] - m_run) : 0.f;
      if (kFp8) {
        __half2 h = __floats2half2_rn(p0, p1);
        const float2 back = __half22float2(h);
        lsum += back.x + back.y;
        pk[c] = *reinterpret_cast<uint32_t*>(&h);
      } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
        const float2 back = __bfloat1622float2(h);
        lsum += back.x + back.y;
        pk[c] = *reinterpret_cast<uint32_t*>(&h);
      }
    }
    l_run += lsum;
    // PV(i-1) done: P buffer is free and O is stable
    if (i >= 1 && !wait_warp(kBarODone, (i - 1) & 1, false)) {
      ok = false;
      break;
    }
    tc_fence_after();
    if (i >= 1 && __any_sync(0xffffffffu, need)) {
      const float a = need ? alpha : 1.f;
      for (int c8 = 0; c8 < 8; ++c8) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * c8, o);
        tmem_wait_ld(o);
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
        tmem_st32(tO + 32 * c8, o);
      }
    }
    tmem_st32(tP, pk);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&sh.bars[kBarPFull]);
  }

  // epilogue: normalised partial output of this CTA's 256 value dims
  const bool have_o = __all_sync(0xffffffffu, ok) && it.n_tiles > 0 &&
                      wait_warp(kBarODone, (it.n_tiles - 1) & 1, false);
  tc_fence_after();
  const int64_t rh = (int64_t)it.b * qrows + qr;
  const int64_t base = ((int64_t)it.k * p.num_splits + it.s) * ((int64_t)R * p.H) + rh;
  const float inv = l_run > 0.f ? kv_scale / l_run : 0.f;
  float* dst = p.part_o + base * kDv + 256 * cta;
  for (int c8 = 0; c8 < 8; ++c8) {
    uint32_t o[32];
    if (have_o) {
      tmem_ld32(tO + 32 * c8, o);
      tmem_wait_ld(o);
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = 0u;
    }
    if (row_ok) {
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        float4 f = make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                               __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
        *reinterpret_cast<float4*>(dst + 32 * c8 + e) = f;
      }
    }
  }
  if (row_ok && cta == 0) {
    p.part_m[base] = l_run > 0.f ? m_run : -INFINITY;
    p.part_l[base] = l_run;
  }
}

template <bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    partial_tc_kernel(const Params p) {
  extern __shared__ unsigned char smem_raw[];
  const Shared sh = carve(smem_raw);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int cta = (int)cluster_ctarank();
  const Item it = decode_item(p, blockIdx.x >> 1);

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sh.bars[kBarKvFull + i], 128);
      mbar_init(&sh.bars[kBarKvEmpty + i], 1);
    }
    mbar_init(&sh.bars[kBarSFull], 1);
    mbar_init(&sh.bars[kBarSFree], 128);
    mbar_init(&sh.bars[kBarPFull], 128);
    mbar_init(&sh.bars[kBarODone], 1);
    mbar_init(&sh.bars[kBarQFull], 128);
    mbar_init(&sh.bars[kBarXFull], 128);
    mbar_init(&sh.bars[kBarXFree], 128);
    mbar_init(&sh.bars[kBarDrain], 1);
    *sh.abort_flag = 0;
    fence_mbarrier_init_cluster();
    const int64_t sb = ((int64_t)it.k * p.batch + it.b) * p.num_splits + it.s;
    const int beg = p.split_beg[sb], end = p.split_end[sb];
    if (cta == 0 && it.t == 0 && (beg < 0 || end < beg || end > p.max_pages))
      raise_status(p.status, DCP_STATUS_BAD_SPLIT);
  }
  if (warp == 8) {
    tmem_alloc(sh.tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tbase = *sh.tmem_slot;

  if (warp < 4) {
    run_softmax<kFp8>(p, sh, it, cta, tbase, tid);
  } else if (warp < 8) {
    run_producer<kFp8>(p, sh, it, cta, tid - 128);
  } else if (tid == 256) {
    run_mma<kFp8>(p, sh, it, cta, tbase);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer no longer touches this CTA's shared memory
  if (warp == 8) {
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
                           float* part_l, uint32_t* status, cudaStream_t stream) {
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
  kern<<<(unsigned)(items * 2), kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dcpmla
