// A verify step for callers that cannot allocate device memory.
//
// The regular entry points leave every intermediate buffer to the caller: the
// row lengths, subpage ids and split bounds of the metadata step, and the
// per-split partial outputs that the merge consumes. Some callers cannot call
// cudaMalloc at all (for example code running inside an allocator callback or a
// runtime that owns the device heap and forbids side allocations). For them,
// dcp_mla_verify_noalloc runs the same three kernels over a fixed scratch area
// that is a file-scope __device__ array of this library: the caller passes only
// inputs and outputs.
//
// The array is kNoAllocScratchBytes (32 MiB) and is held on every GPU that loads
// the library until the process exits. Every call shares it: calls that overlap
// on the GPU (different streams, or different host threads on one device) race
// on it. Nothing in it needs to start at zero (the kernels write every element
// they later read), and it keeps the last call's contents.
#include <mutex>

#include "common.cuh"

namespace dcpmla {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

// Device-side scratch. In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress (per device).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
  size_t row_len, page_ids, split_beg, split_end, part_m, part_l, part_o, order, total;
};

Layout layout_for(const dcp_mla_dims& d, const Derived& x) {
  const size_t nr = d.dcp, B = d.batch, R = x.rows, H = d.num_heads, NS = d.num_splits;
  Layout l;
  size_t off = 0;
  l.row_len = off;
  off += round256(nr * R * sizeof(int32_t));
  l.page_ids = off;
  off += round256(nr * B * x.max_pages * sizeof(int32_t));
  l.split_beg = off;
  off += round256(nr * B * NS * sizeof(int32_t));
  l.split_end = off;
  off += round256(nr * B * NS * sizeof(int32_t));
  l.part_m = off;
  off += round256(nr * NS * R * H * sizeof(float));
  l.part_l = off;
  off += round256(nr * NS * R * H * sizeof(float));
  l.part_o = off;
  off += round256(nr * NS * R * H * kDv * sizeof(float));
  l.order = off;
  off += round256(partial_workspace_bytes(d, (int)nr));
  l.total = off;
  return l;
}

// Device address of the scratch array on the current device, looked up once per
// device (with that device current) and cached.
cudaError_t scratch_address(unsigned char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = ptr;
  }
  *out = static_cast<unsigned char*>(g_scratch_ptr[dev]);
  return cudaSuccess;
}

}  // namespace
}  // namespace dcpmla

using namespace dcpmla;

extern "C" dcp_status dcp_mla_verify_noalloc(const dcp_mla_dims* dims, const int32_t* seq_lens,
                                             const int32_t* block_table, const void* q,
                                             const void* kv, dcp_kv_dtype kv_dtype,
                                             const float* kv_scale, float softmax_scale,
                                             void* out, float* lse, uint32_t* status,
                                             dcp_stream_t stream) {
  dcp_status s = dcp_mla_check_dims(dims, 0, dims ? dims->dcp : 1);
  if (s != DCP_OK) return s;
  if (kv_dtype != DCP_KV_BF16 && kv_dtype != DCP_KV_FP8_E4M3)
    return fail(DCP_ERR_INVALID_ARG, "unknown kv_dtype %d", (int)kv_dtype);
  if (!(softmax_scale > 0.0f) || softmax_scale > 1e30f)
    return fail(DCP_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
  if (dims->batch == 0) return DCP_OK;
  if (!seq_lens || !block_table || !q || !kv || !out || !lse || !status)
    return fail(DCP_ERR_INVALID_ARG, "dcp_mla_verify_noalloc: a required pointer is NULL");
  if (((uintptr_t)q & 15) || ((uintptr_t)kv & 15) || ((uintptr_t)out & 7))
    return fail(DCP_ERR_INVALID_ARG, "q and kv must be 16-byte and out 8-byte aligned");
  const Derived x = derive(*dims);
  const Layout l = layout_for(*dims, x);
  if (l.total > kNoAllocScratchBytes)
    return fail(DCP_ERR_UNSUPPORTED,
                "dcp_mla_verify_noalloc needs %zu bytes of scratch for these dims; its fixed "
                "scratch holds %zu (use the allocating entry points, or fewer splits/rows)",
                l.total, kNoAllocScratchBytes);
  unsigned char* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess)
    return fail(DCP_ERR_CUDA, "scratch set-up failed: %s", cudaGetErrorString(e));
  int32_t* row_len = reinterpret_cast<int32_t*>(base + l.row_len);
  int32_t* page_ids = reinterpret_cast<int32_t*>(base + l.page_ids);
  int32_t* split_beg = reinterpret_cast<int32_t*>(base + l.split_beg);
  int32_t* split_end = reinterpret_cast<int32_t*>(base + l.split_end);
  float* part_m = reinterpret_cast<float*>(base + l.part_m);
  float* part_l = reinterpret_cast<float*>(base + l.part_l);
  float* part_o = reinterpret_cast<float*>(base + l.part_o);
  cudaStream_t st = (cudaStream_t)stream;
  e = launch_metadata(*dims, x, seq_lens, block_table, 0, dims->dcp, row_len, page_ids, split_beg,
                      split_end, status, st);
  if (e == cudaSuccess)
    e = launch_partial(*dims, x, q, kv, kv_dtype, kv_scale, softmax_scale, dims->dcp, row_len,
                       page_ids, split_beg, split_end, part_o, part_m, part_l, base + l.order,
                       status, st);
  if (e == cudaSuccess)
    e = launch_merge(*dims, x, dims->dcp, part_o, part_m, part_l, out, lse, nullptr, status, st);
  if (e != cudaSuccess)
    return fail(DCP_ERR_CUDA, "dcp_mla_verify_noalloc launch failed: %s", cudaGetErrorString(e));
  return DCP_OK;
}
