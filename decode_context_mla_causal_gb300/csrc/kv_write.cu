// The step before the path: the new tokens' latent rows into the rank pools.
//
// "Context Parallel Guide (PCP & DCP)", "How it works" 2: new-token KV is written
// interleaved through a slot mapping that holds -1 for tokens a rank does not
// own; item 4: an FP8 cache carries one per-tensor scale. "Support Kimi-K3 DCP
// with DSpark": global position p lives on rank (p / S) % dcp at local index
// (p / (S*dcp))*S + p % S, i.e. in that rank's block block_table[b][li / bs],
// row li % bs. One thread per (rank, token) forms the mapping; the write moves
// one 576-wide row per block (72 threads x 8 dims).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace dcpmla {
namespace {

constexpr int kMapThreads = 128;
constexpr int kWriteThreads = kDqk / 8;  // 72

__global__ void __launch_bounds__(kMapThreads)
slot_mapping_kernel(int batch, int qlen, int dcp, int interleave, int block_size,
                    int max_blocks_per_seq, int num_blocks, int rank_begin, int num_ranks,
                    const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ block_table,
                    int32_t* __restrict__ slot_mapping, uint32_t* status) {
  const int R = batch * qlen;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)num_ranks * R) return;
  const int k = (int)(idx / R);
  const int row = (int)(idx % R);
  const int b = row / qlen, j = row % qlen;
  const int rank = rank_begin + k;
  const int64_t L = seq_lens[b];
  int32_t slot = -1;
  if (L < qlen) {
    if (k == 0) raise_status(status, DCP_STATUS_BAD_SEQ_LEN);
  } else {
    const int64_t pos = L - qlen + j;
    const int64_t S = interleave, W = dcp;
    if ((pos / S) % W == rank) {
      const int64_t li = (pos / (S * W)) * S + pos % S;
      const int64_t blk_idx = li / block_size;
      if (blk_idx >= max_blocks_per_seq) {
        raise_status(status, DCP_STATUS_LOCAL_OVER_BOUND);
      } else {
        const int32_t blk = block_table[(int64_t)b * max_blocks_per_seq + blk_idx];
        if (blk < 0 || blk >= num_blocks) raise_status(status, DCP_STATUS_BAD_BLOCK_ID);
        else slot = (int32_t)((int64_t)blk * block_size + li % block_size);
      }
    }
  }
  slot_mapping[idx] = slot;
}

// 8 bf16 -> 8 E4M3 codes of x / scale (IEEE fp32 division, RNE, saturated).
__device__ __forceinline__ uint2 quantize8(uint4 x, float scale) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t out[2] = {0u, 0u};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float lo = __uint_as_float(w[e] << 16) / scale;
    const float hi = __uint_as_float(w[e] & 0xFFFF0000u) / scale;
    const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
    out[e >> 1] |= (uint32_t)c << (16 * (e & 1));
  }
  return make_uint2(out[0], out[1]);
}

template <bool kFp8>
__global__ void __launch_bounds__(kWriteThreads)
kv_write_kernel(int rows, int64_t pool_rows, const int32_t* __restrict__ slot_mapping,
                const uint16_t* __restrict__ kv_new, const float* kv_scale, uint8_t* pool,
                uint32_t* status) {
  const int k = blockIdx.y;
  const int row = blockIdx.x;
  const int32_t slot = slot_mapping[(int64_t)k * rows + row];
  if (slot < 0) {
    if (slot != -1 && threadIdx.x == 0) raise_status(status, DCP_STATUS_BAD_PAGE);
    return;
  }
  if (slot >= pool_rows) {
    if (threadIdx.x == 0) raise_status(status, DCP_STATUS_BAD_PAGE);
    return;
  }
  const int d = threadIdx.x * 8;
  const uint4 x = *reinterpret_cast<const uint4*>(kv_new + (int64_t)row * kDqk + d);
  if (kFp8) {
    const float scale = kv_scale ? *kv_scale : 1.0f;
    uint8_t* dst = pool + ((int64_t)k * pool_rows + slot) * kDqk + d;
    *reinterpret_cast<uint2*>(dst) = quantize8(x, scale);
  } else {
    uint8_t* dst = pool + (((int64_t)k * pool_rows + slot) * kDqk + d) * 2;
    *reinterpret_cast<uint4*>(dst) = x;
  }
}

}  // namespace

cudaError_t launch_slot_mapping(const dcp_mla_dims& d, const int32_t* seq_lens,
                                const int32_t* block_table, int rank_begin, int num_ranks,
                                int32_t* slot_mapping, uint32_t* status, cudaStream_t stream) {
  const int64_t n = (int64_t)num_ranks * d.batch * d.qlen;
  if (n == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((n + kMapThreads - 1) / kMapThreads);
  slot_mapping_kernel<<<grid, kMapThreads, 0, stream>>>(
      d.batch, d.qlen, d.dcp, d.interleave, d.block_size, d.max_blocks_per_seq, d.num_blocks,
      rank_begin, num_ranks, seq_lens, block_table, slot_mapping, status);
  return cudaGetLastError();
}

cudaError_t launch_kv_write(const dcp_mla_dims& d, const int32_t* slot_mapping, const void* kv_new,
                            dcp_kv_dtype kv_dtype, const float* kv_scale, int num_ranks,
                            void* pool, uint32_t* status, cudaStream_t stream) {
  const int rows = d.batch * d.qlen;
  if (rows == 0 || num_ranks == 0) return cudaSuccess;
  const dim3 grid((unsigned)rows, (unsigned)num_ranks);
  const int64_t pool_rows = (int64_t)d.num_blocks * d.block_size;
  const uint16_t* src = reinterpret_cast<const uint16_t*>(kv_new);
  uint8_t* dst = reinterpret_cast<uint8_t*>(pool);
  if (kv_dtype == DCP_KV_FP8_E4M3)
    kv_write_kernel<true><<<grid, kWriteThreads, 0, stream>>>(rows, pool_rows, slot_mapping, src,
                                                              kv_scale, dst, status);
  else
    kv_write_kernel<false><<<grid, kWriteThreads, 0, stream>>>(rows, pool_rows, slot_mapping,
                                                               src, kv_scale, dst, status);
  return cudaGetLastError();
}

}  // namespace dcpmla
