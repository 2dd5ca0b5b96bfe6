// C ABI entry points: argument validation, error reporting, launches.
#include <cstdarg>
#include <cstdio>
#include <string>

#include "common.cuh"

namespace dcpmla {

static thread_local std::string g_last_error;

dcp_status fail(dcp_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

static int32_t subpage_of(int32_t block_size) {
  if (block_size <= 0) return -1;
  int32_t low = block_size & (-block_size);
  return low < 128 ? low : 128;
}

Derived derive(const dcp_mla_dims& d) {
  Derived x;
  x.rows = d.batch * d.qlen;
  x.subpage = subpage_of(d.block_size);
  x.ppb = d.block_size / x.subpage;
  x.max_pages = (d.max_local_len + x.subpage - 1) / x.subpage;
  return x;
}

static dcp_status check(const dcp_mla_dims* d, int32_t rank_begin, int32_t num_ranks) {
  g_last_error.clear();
  if (d == nullptr) return fail(DCP_ERR_INVALID_ARG, "dims is NULL");
  if (d->batch < 0) return fail(DCP_ERR_INVALID_ARG, "batch must be >= 0 (got %d)", d->batch);
  if (d->qlen < 1) return fail(DCP_ERR_INVALID_ARG, "qlen must be >= 1 (got %d)", d->qlen);
  if (d->num_heads < 1 || d->num_heads > 1024)
    return fail(DCP_ERR_INVALID_ARG, "num_heads must be in [1, 1024] (got %d)", d->num_heads);
  if (d->dcp < 1) return fail(DCP_ERR_INVALID_ARG, "dcp must be >= 1 (got %d)", d->dcp);
  if (d->block_size < 1)
    return fail(DCP_ERR_INVALID_ARG, "block_size must be >= 1 (got %d)", d->block_size);
  if (d->interleave < 1 || d->interleave > d->block_size)
    return fail(DCP_ERR_INVALID_ARG, "interleave must be in [1, block_size] (got %d)",
                d->interleave);
  if (d->interleave > 1 && d->block_size % d->interleave != 0)
    return fail(DCP_ERR_INVALID_ARG, "block_size %% interleave must be 0 when interleave > 1");
  if (d->max_local_len < 0)
    return fail(DCP_ERR_INVALID_ARG, "max_local_len must be >= 0 (got %d)", d->max_local_len);
  if (d->max_blocks_per_seq < 1)
    return fail(DCP_ERR_INVALID_ARG, "max_blocks_per_seq must be >= 1");
  if ((int64_t)d->max_blocks_per_seq * d->block_size < (int64_t)d->max_local_len)
    return fail(DCP_ERR_INVALID_ARG,
                "max_blocks_per_seq * block_size (%lld) must cover max_local_len (%d)",
                (long long)d->max_blocks_per_seq * d->block_size, d->max_local_len);
  if (d->num_blocks < 1) return fail(DCP_ERR_INVALID_ARG, "num_blocks must be >= 1");
  if ((int64_t)d->num_blocks * d->block_size > (int64_t)INT32_MAX)
    return fail(DCP_ERR_UNSUPPORTED, "num_blocks * block_size must fit in int32");
  if (d->num_splits < 1 || d->num_splits > 4096)
    return fail(DCP_ERR_INVALID_ARG, "num_splits must be in [1, 4096] (got %d)", d->num_splits);
  if (d->causal != 0 && d->causal != 1)
    return fail(DCP_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (d->base_splits < 0 || d->base_splits > d->num_splits)
    return fail(DCP_ERR_INVALID_ARG, "base_splits must be in [0, num_splits=%d] (got %d)",
                d->num_splits, d->base_splits);
  if (d->base_splits > 0 && d->base_splits < d->num_splits &&
      (int64_t)d->batch * d->dcp > kBalanceMaxPairs)
    return fail(DCP_ERR_UNSUPPORTED, "wave balancing takes at most %d (rank, sequence) pairs",
                kBalanceMaxPairs);
  if ((int64_t)d->batch * d->qlen * d->num_heads > (int64_t)(1 << 24))
    return fail(DCP_ERR_UNSUPPORTED, "batch*qlen*num_heads above 2^24");
  if (rank_begin < 0 || num_ranks < 1 || (int64_t)rank_begin + num_ranks > d->dcp)
    return fail(DCP_ERR_INVALID_ARG, "rank range [%d, %d) outside [0, dcp=%d)", rank_begin,
                rank_begin + num_ranks, d->dcp);
  return DCP_OK;
}

static dcp_status launched(cudaError_t e, const char* what) {
  if (e != cudaSuccess)
    return fail(DCP_ERR_CUDA, "%s launch failed: %s", what, cudaGetErrorString(e));
  return DCP_OK;
}

}  // namespace dcpmla

using namespace dcpmla;

extern "C" {

int32_t dcp_mla_subpage_size(int32_t block_size) { return subpage_of(block_size); }

int32_t dcp_mla_max_pages(const dcp_mla_dims* dims) {
  if (check(dims, 0, dims ? (dims->dcp > 0 ? dims->dcp : 1) : 1) != DCP_OK) return -1;
  return derive(*dims).max_pages;
}

dcp_status dcp_mla_check_dims(const dcp_mla_dims* dims, int32_t rank_begin, int32_t num_ranks) {
  return check(dims, rank_begin, num_ranks);
}

dcp_status dcp_mla_metadata(const dcp_mla_dims* dims, const int32_t* seq_lens,
                            const int32_t* block_table, int32_t rank_begin, int32_t num_ranks,
                            int32_t* row_len, int32_t* page_ids, int32_t* split_beg,
                            int32_t* split_end, uint32_t* status, dcp_stream_t stream) {
  dcp_status s = check(dims, rank_begin, num_ranks);
  if (s != DCP_OK) return s;
  if (dims->batch == 0) return DCP_OK;
  if (!seq_lens || !block_table || !row_len || !page_ids || !split_beg || !split_end || !status)
    return fail(DCP_ERR_INVALID_ARG, "dcp_mla_metadata: a required pointer is NULL");
  Derived x = derive(*dims);
  return launched(launch_metadata(*dims, x, seq_lens, block_table, rank_begin, num_ranks,
                                  row_len, page_ids, split_beg, split_end, status,
                                  (cudaStream_t)stream),
                  "dcp_mla_metadata");
}

static dcp_status partial_call(const dcp_mla_dims* dims, const void* q, const void* kv,
                               dcp_kv_dtype kv_dtype, const float* kv_scale, float softmax_scale,
                               int32_t rank_begin, int32_t num_ranks, const int32_t* row_len,
                               const int32_t* page_ids, const int32_t* split_beg,
                               const int32_t* split_end, float* part_o, float* part_m,
                               float* part_l, void* workspace, uint32_t* status,
                               dcp_stream_t stream, uint64_t hold_q_ns, const char* what) {
  dcp_status s = check(dims, rank_begin, num_ranks);
  if (s != DCP_OK) return s;
  if (kv_dtype != DCP_KV_BF16 && kv_dtype != DCP_KV_FP8_E4M3)
    return fail(DCP_ERR_INVALID_ARG, "unknown kv_dtype %d", (int)kv_dtype);
  if (!(softmax_scale > 0.0f) || softmax_scale > 1e30f)
    return fail(DCP_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
  if (dims->batch == 0) return DCP_OK;
  if (!q || !kv || !row_len || !page_ids || !split_beg || !split_end || !part_o || !part_m ||
      !part_l || !status)
    return fail(DCP_ERR_INVALID_ARG, "%s: a required pointer is NULL", what);
  if (((uintptr_t)q & 15) || ((uintptr_t)kv & 15) || ((uintptr_t)part_o & 15) ||
      ((uintptr_t)workspace & 15))
    return fail(DCP_ERR_INVALID_ARG, "q, kv, part_o and workspace must be 16-byte aligned");
  Derived x = derive(*dims);
  return launched(launch_partial(*dims, x, q, kv, kv_dtype, kv_scale, softmax_scale, num_ranks,
                                 row_len, page_ids, split_beg, split_end, part_o, part_m, part_l,
                                 workspace, status, (cudaStream_t)stream, nullptr, hold_q_ns),
                  what);
}

dcp_status dcp_mla_partial(const dcp_mla_dims* dims, const void* q, const void* kv,
                           dcp_kv_dtype kv_dtype, const float* kv_scale, float softmax_scale,
                           int32_t rank_begin, int32_t num_ranks, const int32_t* row_len,
                           const int32_t* page_ids, const int32_t* split_beg,
                           const int32_t* split_end, float* part_o, float* part_m,
                           float* part_l, void* workspace, uint32_t* status,
                           dcp_stream_t stream) {
  return partial_call(dims, q, kv, kv_dtype, kv_scale, softmax_scale, rank_begin, num_ranks,
                      row_len, page_ids, split_beg, split_end, part_o, part_m, part_l, workspace,
                      status, stream, 0, "dcp_mla_partial");
}

dcp_status dcp_mla_partial_hold_q(const dcp_mla_dims* dims, const void* q, const void* kv,
                                  dcp_kv_dtype kv_dtype, const float* kv_scale,
                                  float softmax_scale, int32_t rank_begin, int32_t num_ranks,
                                  const int32_t* row_len, const int32_t* page_ids,
                                  const int32_t* split_beg, const int32_t* split_end,
                                  float* part_o, float* part_m, float* part_l, void* workspace,
                                  uint32_t* status, uint64_t q_wait_ns, dcp_stream_t stream) {
  if (q_wait_ns == 0 || q_wait_ns > 4000000000ull)
    return fail(DCP_ERR_INVALID_ARG, "q_wait_ns must be in (0, 4e9] (got %llu)",
                (unsigned long long)q_wait_ns);
  return partial_call(dims, q, kv, kv_dtype, kv_scale, softmax_scale, rank_begin, num_ranks,
                      row_len, page_ids, split_beg, split_end, part_o, part_m, part_l, workspace,
                      status, stream, q_wait_ns, "dcp_mla_partial_hold_q");
}

dcp_status dcp_mla_partial_packed(const dcp_mla_dims* dims, const void* q, const void* kv,
                                  dcp_kv_dtype kv_dtype, const float* kv_scale,
                                  float softmax_scale, int32_t rank_begin, int32_t num_ranks,
                                  const int32_t* row_len, const int32_t* page_ids,
                                  const int32_t* split_beg, const int32_t* split_end,
                                  void* send, void* workspace, uint32_t* status,
                                  dcp_stream_t stream) {
  dcp_status s = check(dims, rank_begin, num_ranks);
  if (s != DCP_OK) return s;
  if (dims->num_splits != 1)
    return fail(DCP_ERR_UNSUPPORTED, "dcp_mla_partial_packed needs num_splits == 1 (got %d)",
                dims->num_splits);
  if (dims->num_heads % dims->dcp != 0)
    return fail(DCP_ERR_UNSUPPORTED, "num_heads (%d) must be a multiple of dcp (%d)",
                dims->num_heads, dims->dcp);
  if (kv_dtype != DCP_KV_BF16 && kv_dtype != DCP_KV_FP8_E4M3)
    return fail(DCP_ERR_INVALID_ARG, "unknown kv_dtype %d", (int)kv_dtype);
  if (!(softmax_scale > 0.0f) || softmax_scale > 1e30f)
    return fail(DCP_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
  if (dims->batch == 0) return DCP_OK;
  if (!q || !kv || !row_len || !page_ids || !split_beg || !split_end || !send || !status)
    return fail(DCP_ERR_INVALID_ARG, "dcp_mla_partial_packed: a required pointer is NULL");
  if (((uintptr_t)q & 15) || ((uintptr_t)kv & 15) || ((uintptr_t)send & 15) ||
      ((uintptr_t)workspace & 15))
    return fail(DCP_ERR_INVALID_ARG, "q, kv, send and workspace must be 16-byte aligned");
  Derived x = derive(*dims);
  return launched(launch_partial(*dims, x, q, kv, kv_dtype, kv_scale, softmax_scale, num_ranks,
                                 row_len, page_ids, split_beg, split_end, nullptr, nullptr,
                                 nullptr, workspace, status, (cudaStream_t)stream, send),
                  "dcp_mla_partial_packed");
}

dcp_status dcp_mla_workspace_size(const dcp_mla_dims* dims, int32_t num_ranks, size_t* bytes) {
  dcp_status s = check(dims, 0, num_ranks);
  if (s != DCP_OK) return s;
  if (bytes == nullptr) return fail(DCP_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = partial_workspace_bytes(*dims, num_ranks);
  return DCP_OK;
}

dcp_status dcp_lse_merge(const dcp_mla_dims* dims, int32_t num_ranks, const float* part_o,
                         const float* part_m, const float* part_l, void* out, float* lse,
                         float* rank_lse, uint32_t* status, dcp_stream_t stream) {
  dcp_status s = check(dims, 0, num_ranks);
  if (s != DCP_OK) return s;
  if (dims->batch == 0) return DCP_OK;
  if (!part_o || !part_m || !part_l || !out || !lse || !status)
    return fail(DCP_ERR_INVALID_ARG, "dcp_lse_merge: a required pointer is NULL");
  if (((uintptr_t)part_o & 15) || ((uintptr_t)out & 7))
    return fail(DCP_ERR_INVALID_ARG, "part_o must be 16-byte and out 8-byte aligned");
  Derived x = derive(*dims);
  return launched(launch_merge(*dims, x, num_ranks, part_o, part_m, part_l, out, lse, rank_lse,
                               status, (cudaStream_t)stream),
                  "dcp_lse_merge");
}

dcp_status dcp_kv_slot_mapping(const dcp_mla_dims* dims, const int32_t* seq_lens,
                               const int32_t* block_table, int32_t rank_begin, int32_t num_ranks,
                               int32_t* slot_mapping, uint32_t* status, dcp_stream_t stream) {
  dcp_status s = check(dims, rank_begin, num_ranks);
  if (s != DCP_OK) return s;
  if (dims->batch == 0 || num_ranks == 0) return DCP_OK;
  if (!seq_lens || !block_table || !slot_mapping || !status)
    return fail(DCP_ERR_INVALID_ARG, "dcp_kv_slot_mapping: a required pointer is NULL");
  return launched(launch_slot_mapping(*dims, seq_lens, block_table, rank_begin, num_ranks,
                                      slot_mapping, status, (cudaStream_t)stream),
                  "dcp_kv_slot_mapping");
}

dcp_status dcp_kv_write(const dcp_mla_dims* dims, const int32_t* slot_mapping, const void* kv_new,
                        dcp_kv_dtype kv_dtype, const float* kv_scale, int32_t num_ranks,
                        void* pool, uint32_t* status, dcp_stream_t stream) {
  dcp_status s = check(dims, 0, num_ranks);
  if (s != DCP_OK) return s;
  if (kv_dtype != DCP_KV_BF16 && kv_dtype != DCP_KV_FP8_E4M3)
    return fail(DCP_ERR_INVALID_ARG, "unknown kv_dtype %d", (int)kv_dtype);
  if (dims->batch == 0 || num_ranks == 0) return DCP_OK;
  if (!slot_mapping || !kv_new || !pool || !status)
    return fail(DCP_ERR_INVALID_ARG, "dcp_kv_write: a required pointer is NULL");
  if (((uintptr_t)kv_new & 15) || ((uintptr_t)pool & 15))
    return fail(DCP_ERR_INVALID_ARG, "kv_new and pool must be 16-byte aligned");
  return launched(launch_kv_write(*dims, slot_mapping, kv_new, kv_dtype, kv_scale, num_ranks,
                                  pool, status, (cudaStream_t)stream),
                  "dcp_kv_write");
}

int64_t dcp_a2a_chunk_words(const dcp_mla_dims* dims, int32_t payload) {
  if (check(dims, 0, 1) != DCP_OK) return -1;
  if (payload < 1 || payload > kDv || dims->num_heads % dims->dcp != 0) return -1;
  return dcpmla::a2a_chunk_words(dims->batch * dims->qlen, dims->num_heads / dims->dcp, payload);
}

dcp_status dcp_a2a_pack(const dcp_mla_dims* dims, int32_t num_ranks, const float* part_o,
                        const float* part_m, const float* part_l, void* send, uint32_t* status,
                        dcp_stream_t stream) {
  (void)status;
  dcp_status s = check(dims, 0, num_ranks);
  if (s != DCP_OK) return s;
  if (dims->num_heads % dims->dcp != 0)
    return fail(DCP_ERR_INVALID_ARG, "num_heads (%d) must be a multiple of dcp (%d)",
                dims->num_heads, dims->dcp);
  if (dims->batch == 0) return DCP_OK;
  if (!part_o || !part_m || !part_l || !send)
    return fail(DCP_ERR_INVALID_ARG, "dcp_a2a_pack: a required pointer is NULL");
  if (((uintptr_t)part_o & 15) || ((uintptr_t)send & 15))
    return fail(DCP_ERR_INVALID_ARG, "part_o and send must be 16-byte aligned");
  Derived x = derive(*dims);
  return launched(launch_a2a_pack(*dims, x, num_ranks, part_o, part_m, part_l, send,
                                  (cudaStream_t)stream),
                  "dcp_a2a_pack");
}

dcp_status dcp_a2a_project(const dcp_mla_dims* dims, int32_t num_ranks, const void* send,
                           const void* w_v, int32_t payload, void* send_projected,
                           uint32_t* status, dcp_stream_t stream) {
  dcp_status s = check(dims, 0, num_ranks);
  if (s != DCP_OK) return s;
  if (dims->num_heads % dims->dcp != 0)
    return fail(DCP_ERR_INVALID_ARG, "num_heads (%d) must be a multiple of dcp (%d)",
                dims->num_heads, dims->dcp);
  if (payload < 16 || payload > 256 || payload % 16 != 0)
    return fail(DCP_ERR_INVALID_ARG, "projected payload must be a multiple of 16 in [16, 256]");
  if (dims->batch == 0) return DCP_OK;
  if (!send || !w_v || !send_projected)
    return fail(DCP_ERR_INVALID_ARG, "dcp_a2a_project: a required pointer is NULL");
  if (((uintptr_t)send & 15) || ((uintptr_t)w_v & 15) || ((uintptr_t)send_projected & 15))
    return fail(DCP_ERR_INVALID_ARG, "send, w_v and send_projected must be 16-byte aligned");
  Derived x = derive(*dims);
  return launched(launch_a2a_project(*dims, x, num_ranks, send, w_v, payload, send_projected,
                                     status, (cudaStream_t)stream),
                  "dcp_a2a_project");
}

dcp_status dcp_a2a_combine(const dcp_mla_dims* dims, int32_t payload, const void* recv,
                           int64_t src_stride, int64_t dst_stride, int32_t dst_begin,
                           int32_t num_dst, void* out, float* lse, uint32_t* status,
                           dcp_stream_t stream) {
  (void)status;
  dcp_status s = check(dims, dst_begin, num_dst);
  if (s != DCP_OK) return s;
  if (dims->num_heads % dims->dcp != 0)
    return fail(DCP_ERR_INVALID_ARG, "num_heads (%d) must be a multiple of dcp (%d)",
                dims->num_heads, dims->dcp);
  if (payload < 4 || payload > kDv || payload % 4 != 0)
    return fail(DCP_ERR_INVALID_ARG, "payload must be a multiple of 4 in [4, 512]");
  if (src_stride < 0 || dst_stride < 0 || (src_stride & 7) || (dst_stride & 7))
    return fail(DCP_ERR_INVALID_ARG, "strides must be non-negative multiples of 8 words");
  if (dims->batch == 0) return DCP_OK;
  if (!recv || !out || !lse)
    return fail(DCP_ERR_INVALID_ARG, "dcp_a2a_combine: a required pointer is NULL");
  if (((uintptr_t)recv & 15) || ((uintptr_t)out & 7))
    return fail(DCP_ERR_INVALID_ARG, "recv must be 16-byte and out 8-byte aligned");
  Derived x = derive(*dims);
  return launched(launch_a2a_combine(*dims, x, payload, recv, src_stride, dst_stride, dst_begin,
                                     num_dst, out, lse, (cudaStream_t)stream),
                  "dcp_a2a_combine");
}

int32_t dcp_mla_concurrent_items(void) { return partial_concurrent_items(); }

const char* dcp_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
