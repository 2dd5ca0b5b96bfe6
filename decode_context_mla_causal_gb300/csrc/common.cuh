// Shared definitions of the CUDA library (not shared with the CPU oracle).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dcp_mla.h"

namespace dcpmla {

constexpr int kDqk = DCP_MLA_QK_DIM;  // 576
constexpr int kDv = DCP_MLA_V_DIM;    // 512

// Host-side derived sizes of a dims struct (validated by check_dims first).
struct Derived {
  int rows;       // R = batch * qlen
  int subpage;    // P
  int ppb;        // subpages per block
  int max_pages;  // MP
};

Derived derive(const dcp_mla_dims& d);

// Record a message for dcp_last_error() and return the status.
dcp_status fail(dcp_status s, const char* fmt, ...);

// Internal launchers (argument checks already done by the API layer).
cudaError_t launch_metadata(const dcp_mla_dims& d, const Derived& x, const int32_t* seq_lens,
                            const int32_t* block_table, int rank_begin, int num_ranks,
                            int32_t* row_len, int32_t* page_ids, int32_t* split_beg,
                            int32_t* split_end, uint32_t* status, cudaStream_t stream);

cudaError_t launch_partial(const dcp_mla_dims& d, const Derived& x, const void* q,
                           const void* kv, dcp_kv_dtype kv_dtype, const float* kv_scale,
                           float softmax_scale, int num_ranks, const int32_t* row_len,
                           const int32_t* page_ids, const int32_t* split_beg,
                           const int32_t* split_end, float* part_o, float* part_m,
                           float* part_l, void* workspace, uint32_t* status,
                           cudaStream_t stream, void* send = nullptr,
                           uint64_t hold_q_ns = 0);

// Device workspace launch_partial uses for the item order (bytes, 16-byte multiple).
size_t partial_workspace_bytes(const dcp_mla_dims& d, int num_ranks);

// Clusters of the partial kernel the current device runs at once (cached per
// device), or a negative value when the query fails.
int partial_concurrent_items();

// Wave balancing reads every (rank, sequence) pair's length in each metadata CTA.
constexpr int kBalanceMaxPairs = 1 << 16;

// Tiles of 64 tokens per work item, the unit of the split plan.
constexpr int kPlanTileTokens = 64;
// Wave balancing cuts no piece below this many tiles.
constexpr int kPlanMinPieceTiles = 8;

cudaError_t launch_merge(const dcp_mla_dims& d, const Derived& x, int num_ranks,
                         const float* part_o, const float* part_m, const float* part_l,
                         void* out, float* lse, float* rank_lse, uint32_t* status,
                         cudaStream_t stream);

cudaError_t launch_slot_mapping(const dcp_mla_dims& d, const int32_t* seq_lens,
                                const int32_t* block_table, int rank_begin, int num_ranks,
                                int32_t* slot_mapping, uint32_t* status, cudaStream_t stream);

cudaError_t launch_kv_write(const dcp_mla_dims& d, const int32_t* slot_mapping, const void* kv_new,
                            dcp_kv_dtype kv_dtype, const float* kv_scale, int num_ranks,
                            void* pool, uint32_t* status, cudaStream_t stream);

int64_t a2a_chunk_words(int R, int Hg, int P);

cudaError_t launch_a2a_pack(const dcp_mla_dims& d, const Derived& x, int num_ranks,
                            const float* part_o, const float* part_m, const float* part_l,
                            void* send, cudaStream_t stream);

cudaError_t launch_a2a_project(const dcp_mla_dims& d, const Derived& x, int num_ranks,
                               const void* send_in, const void* w_v, int payload, void* send,
                               uint32_t* status, cudaStream_t stream);

cudaError_t launch_a2a_combine(const dcp_mla_dims& d, const Derived& x, int payload,
                               const void* recv, int64_t src_stride, int64_t dst_stride,
                               int dst_begin, int num_dst, void* out, float* lse,
                               cudaStream_t stream);

__device__ __forceinline__ void raise_status(uint32_t* status, uint32_t bits) {
  if (status != nullptr) atomicOr(status, bits);
}

}  // namespace dcpmla
