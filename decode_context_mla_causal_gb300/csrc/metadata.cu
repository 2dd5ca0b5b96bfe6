// Steps 1+2: per-row rank-local lengths, subpage ids and split bounds.
//
// "Support Kimi-K3 DCP with DSpark" (review thread) gives the local length of a
// row with global boundary g on rank r of an interleaved shard; "[ROCm][MLA][DCP]
// Support causal multi-token verification" (Implementation, items 1, 2, 5) maps
// each verify row's causal boundary through it, expands blocks into bounded
// subpages and lays the metadata out at a static bound. One CTA per
// (rank, sequence); every output element is written, padding included, so a
// graph replay never sees stale entries.
//
// Split plan. Without wave balancing every (rank, sequence) pair takes NS equal
// splits. With it (0 < base_splits < NS) a pair takes base_splits, except the
// shortest pairs whose items would run in a part-filled last wave: those share
// that wave's C slots (C = clusters the partial kernel runs at once). A CTA finds
// its pair's place in the length order by counting, over all dcp*batch pairs
// (lengths from seq_lens, as the longest row's local length), the longer ones and
// the equal ones before it; no sort, and the same answer in a per-rank call.
#include "common.cuh"

namespace dcpmla {
namespace {

constexpr int kMetaThreads = 256;

// Local length of a row whose global causal boundary is g, on `rank`
// ("Support Kimi-K3 DCP with DSpark", review thread), unclamped.
__device__ __forceinline__ int64_t local_len(int64_t g, int rank, int64_t span, int interleave) {
  if (g <= 0) return 0;
  int64_t rem = g % span - (int64_t)rank * interleave;
  rem = rem < 0 ? 0 : (rem > interleave ? interleave : rem);
  return g / span * interleave + rem;
}

// Tiles of the longest row of (rank, sequence of global length L): its boundary is L
// whether causal or not.
__device__ __forceinline__ int pair_tiles(int64_t L, int rank, int64_t span, int interleave,
                                          int max_local_len) {
  int64_t loc = local_len(L < 0 ? 0 : L, rank, span, interleave);
  if (loc > max_local_len) loc = max_local_len;
  return (int)((loc + kPlanTileTokens - 1) / kPlanTileTokens);
}

// Block-wide sum of three counters (every thread gets the totals).
__device__ __forceinline__ void block_sum3(int& a, int& b, int& c, int* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
    c += __shfl_xor_sync(0xffffffffu, c, o);
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0) {
    scratch[3 * wid] = a;
    scratch[3 * wid + 1] = b;
    scratch[3 * wid + 2] = c;
  }
  __syncthreads();
  a = b = c = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    a += scratch[3 * w];
    b += scratch[3 * w + 1];
    c += scratch[3 * w + 2];
  }
}

// Splits of pair (rank, b) under wave balancing; base_splits when it is not a
// pair of the last wave (every thread of the block returns the same value).
__device__ int balanced_splits(int rank, int b, int batch, int dcp, int64_t span,
                               int interleave, int max_local_len, int row_tiles, int base,
                               int num_splits, int concurrent, const int32_t* seq_lens,
                               int* scratch) {
  const int me = rank * batch + b;  // rank-major pair index
  const int t_me = pair_tiles(seq_lens[b], rank, span, interleave, max_local_len);
  int longer = 0, equal_before = 0, live = 0;
  const int pairs = dcp * batch;
  for (int v = threadIdx.x; v < pairs; v += blockDim.x) {
    const int r = v / batch, bb = v - r * batch;
    const int t = pair_tiles(seq_lens[bb], r, span, interleave, max_local_len);
    longer += t > t_me;
    equal_before += (t == t_me && v < me);
    live += t > 0;
  }
  block_sum3(longer, equal_before, live, scratch);
  if (t_me == 0) return 1;
  const int64_t per = (int64_t)row_tiles * base;  // items of one pair
  const int64_t C = concurrent;
  const int64_t rem = (int64_t)live * per % C;
  if (rem == 0 || 2 * rem > C) return base;
  const int64_t tail = (rem + per - 1) / per;  // pairs of the last wave
  const int64_t pos = longer + equal_before;   // 0 = longest
  if (pos < live - tail) return base;
  const int64_t j = pos - (live - tail);
  const int64_t kf = C / (tail * per);
  const int64_t hi = (C - kf * tail * per) / per;
  int64_t s = (int64_t)base * ((kf > 1 ? kf : 1) + (j < hi ? 1 : 0));
  if (s > num_splits) s = num_splits;
  const int64_t by_len = t_me / kPlanMinPieceTiles;
  if (s > by_len) s = by_len;
  return (int)(s > base ? s : base);
}

__global__ void __launch_bounds__(kMetaThreads)
metadata_kernel(int batch, int qlen, int dcp, int interleave, int max_local_len,
                int max_blocks_per_seq, int num_blocks, int num_splits, int causal,
                int subpage, int ppb, int max_pages, const int32_t* __restrict__ seq_lens,
                const int32_t* __restrict__ block_table, int rank_begin,
                int32_t* __restrict__ row_len, int32_t* __restrict__ page_ids,
                int32_t* __restrict__ split_beg, int32_t* __restrict__ split_end,
                uint32_t* status, int row_tiles, int base_splits, int concurrent) {
  const int b = blockIdx.x;
  const int k = blockIdx.y;  // rank index inside the call
  const int rank = rank_begin + k;
  __shared__ int s_longest;
  __shared__ uint32_t s_status;
  __shared__ int s_scratch[3 * (kMetaThreads / 32)];
  if (threadIdx.x == 0) {
    s_longest = 0;
    s_status = 0;
  }
  __syncthreads();

  const int64_t L = seq_lens[b];
  if (threadIdx.x == 0 && (L < 0 || (causal && L < qlen))) atomicOr(&s_status, DCP_STATUS_BAD_SEQ_LEN);
  const int64_t span = (int64_t)dcp * interleave;
  for (int j = threadIdx.x; j < qlen; j += blockDim.x) {
    const int64_t g = causal ? L - qlen + 1 + j : L;  // global causal boundary of row j
    int64_t local = local_len(g, rank, span, interleave);
    if (local > max_local_len) {
      atomicOr(&s_status, DCP_STATUS_LOCAL_OVER_BOUND);
      local = max_local_len;
    }
    row_len[(int64_t)k * batch * qlen + (int64_t)b * qlen + j] = (int32_t)local;
    atomicMax(&s_longest, (int)local);
  }
  __syncthreads();
  const int npages = (s_longest + subpage - 1) / subpage;
  int32_t* pages = page_ids + ((int64_t)k * batch + b) * max_pages;
  const int32_t* table = block_table + (int64_t)b * max_blocks_per_seq;
  for (int p = threadIdx.x; p < max_pages; p += blockDim.x) {
    int32_t id = -1;
    if (p < npages) {
      const int bi = p / ppb;
      const int32_t blk = bi < max_blocks_per_seq ? table[bi] : -1;
      if (blk >= 0 && blk < num_blocks) {
        id = blk * ppb + p % ppb;
      } else {
        atomicOr(&s_status, DCP_STATUS_BAD_BLOCK_ID);
      }
    }
    pages[p] = id;
  }
  const int n = base_splits > 0 && base_splits < num_splits
                    ? balanced_splits(rank, b, batch, dcp, span, interleave, max_local_len,
                                      row_tiles, base_splits, num_splits, concurrent, seq_lens,
                                      s_scratch)
                    : num_splits;
  int32_t* beg = split_beg + ((int64_t)k * batch + b) * num_splits;
  int32_t* end = split_end + ((int64_t)k * batch + b) * num_splits;
  for (int s = threadIdx.x; s < num_splits; s += blockDim.x) {
    beg[s] = (int32_t)(s < n ? ((int64_t)s * npages) / n : npages);
    end[s] = (int32_t)(s < n ? ((int64_t)(s + 1) * npages) / n : npages);
  }
  __syncthreads();
  if (threadIdx.x == 0 && s_status) raise_status(status, s_status);
}

}  // namespace

cudaError_t launch_metadata(const dcp_mla_dims& d, const Derived& x, const int32_t* seq_lens,
                            const int32_t* block_table, int rank_begin, int num_ranks,
                            int32_t* row_len, int32_t* page_ids, int32_t* split_beg,
                            int32_t* split_end, uint32_t* status, cudaStream_t stream) {
  int concurrent = 1;
  const bool balance = d.base_splits > 0 && d.base_splits < d.num_splits;
  if (balance) {
    concurrent = partial_concurrent_items();
    if (concurrent < 1) return cudaErrorInvalidConfiguration;
  }
  dim3 grid(d.batch, num_ranks);
  metadata_kernel<<<grid, kMetaThreads, 0, stream>>>(
      d.batch, d.qlen, d.dcp, d.interleave, d.max_local_len, d.max_blocks_per_seq, d.num_blocks,
      d.num_splits, d.causal, x.subpage, x.ppb, x.max_pages, seq_lens, block_table, rank_begin,
      row_len, page_ids, split_beg, split_end, status, (d.qlen * d.num_heads + 127) / 128,
      balance ? d.base_splits : 0, concurrent);
  return cudaGetLastError();
}

}  // namespace dcpmla
