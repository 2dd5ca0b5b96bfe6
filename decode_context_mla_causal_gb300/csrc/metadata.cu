// Steps 1+2: per-row rank-local lengths, subpage ids and split bounds.
//
// "Support Kimi-K3 DCP with DSpark" (review thread) gives the local length of a
// row with global boundary g on rank r of an interleaved shard; "[ROCm][MLA][DCP]
// Support causal multi-token verification" (Implementation, items 1, 2, 5) maps
// each verify row's causal boundary through it, expands blocks into bounded
// subpages and lays the metadata out at a static bound. One CTA per
// (rank, sequence); every output element is written, padding included, so a
// graph replay never sees stale entries.
#include "common.cuh"

namespace dcpmla {
namespace {

constexpr int kMetaThreads = 256;

__global__ void __launch_bounds__(kMetaThreads)
metadata_kernel(int batch, int qlen, int dcp, int interleave, int max_local_len,
                int max_blocks_per_seq, int num_blocks, int num_splits, int causal,
                int subpage, int ppb, int max_pages, const int32_t* __restrict__ seq_lens,
                const int32_t* __restrict__ block_table, int rank_begin,
                int32_t* __restrict__ row_len, int32_t* __restrict__ page_ids,
                int32_t* __restrict__ split_beg, int32_t* __restrict__ split_end,
                uint32_t* status) {
  const int b = blockIdx.x;
  const int k = blockIdx.y;  // rank index inside the call
  const int rank = rank_begin + k;
  __shared__ int s_longest;
  __shared__ uint32_t s_status;
  if (threadIdx.x == 0) {
    s_longest = 0;
    s_status = 0;
  }
  __syncthreads();

  const int64_t L = seq_lens[b];
  if (threadIdx.x == 0 && (L < 0 || (causal && L < qlen))) atomicOr(&s_status, DCP_STATUS_BAD_SEQ_LEN);
  const int64_t span = (int64_t)dcp * interleave;
  for (int j = threadIdx.x; j < qlen; j += blockDim.x) {
    int64_t g = causal ? L - qlen + 1 + j : L;  // global causal boundary of row j
    int64_t local = 0;
    if (g > 0) {
      int64_t rem = g % span - (int64_t)rank * interleave;
      rem = rem < 0 ? 0 : (rem > interleave ? interleave : rem);
      local = g / span * interleave + rem;
    }
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
  int32_t* beg = split_beg + ((int64_t)k * batch + b) * num_splits;
  int32_t* end = split_end + ((int64_t)k * batch + b) * num_splits;
  for (int s = threadIdx.x; s < num_splits; s += blockDim.x) {
    beg[s] = (int32_t)(((int64_t)s * npages) / num_splits);
    end[s] = (int32_t)(((int64_t)(s + 1) * npages) / num_splits);
  }
  __syncthreads();
  if (threadIdx.x == 0 && s_status) raise_status(status, s_status);
}

}  // namespace

cudaError_t launch_metadata(const dcp_mla_dims& d, const Derived& x, const int32_t* seq_lens,
                            const int32_t* block_table, int rank_begin, int num_ranks,
                            int32_t* row_len, int32_t* page_ids, int32_t* split_beg,
                            int32_t* split_end, uint32_t* status, cudaStream_t stream) {
  dim3 grid(d.batch, num_ranks);
  metadata_kernel<<<grid, kMetaThreads, 0, stream>>>(
      d.batch, d.qlen, d.dcp, d.interleave, d.max_local_len, d.max_blocks_per_seq, d.num_blocks,
      d.num_splits, d.causal, x.subpage, x.ppb, x.max_pages, seq_lens, block_table, rank_begin,
      row_len, page_ids, split_beg, split_end, status);
  return cudaGetLastError();
}

}  // namespace dcpmla
