/*
 * dcp_mla.h -- C ABI of libdcpmla.so: decode-context-parallel (DCP) causal
 * multi-token MLA verification attention over a paged latent KV cache, for
 * NVIDIA GB300 (sm_103a).
 *
 * The method (sources are named by page title and section):
 *
 *   "Context Parallel Guide (PCP & DCP)" -- Decode Context Parallel (DCP) Guide.
 *     The latent KV cache is sharded by sequence position over `dcp` ranks:
 *     token p lives on rank (p / S) % dcp (S = interleave_size), at rank-local
 *     index (p / (S*dcp))*S + p % S ("--dcp-config" table, "interleave_size").
 *     One block-table entry is shared by all ranks and names, on each rank, that
 *     rank's own physical block of block_size local tokens ("How it works" 1).
 *     Each rank attends its local KV and returns its LSE; the partial outputs are
 *     LSE-corrected and summed ("Decode"). FP8 caches use one per-tensor scale.
 *   "Support Kimi-K3 DCP with DSpark" -- review thread: the rank-local length of
 *     a row with global boundary g is
 *       g/(dcp*S)*S + clamp(g % (dcp*S) - rank*S, 0, S).
 *   "[ROCm][MLA][DCP] Support causal multi-token verification" -- Implementation:
 *     (1) each verification row's global causal boundary is mapped to its
 *     rank-local KV length; (2) physical blocks are expanded into bounded
 *     subpages; (3) split-KV MLA emits unreduced partial outputs with base-2
 *     max/sum statistics, later turned into natural-log LSE; (4) an LSE merge
 *     produces the BF16 output. Row metadata is laid out at a static maximum
 *     local bound so that the launches can be captured in a CUDA graph.
 *
 * Readings this library takes where the pages are silent:
 *   - seq_lens[b] counts every token of sequence b INCLUDING its qlen verify
 *     tokens, whose latent rows are already in the cache; verify row j (0-based)
 *     attends global positions [0, g_j) with g_j = seq_lens[b] - qlen + 1 + j.
 *     With dims.causal == 0 every row attends [0, seq_lens[b]) (the
 *     bidirectional DSpark draft block of "DCP + Speculative Decode").
 *   - Absorbed MLA: q and k are 576 wide (512 latent + 64 rope); v is the first
 *     512 dims of the same cache row.
 *   - Subpage size P = min(128, largest power of two dividing block_size);
 *     subpage p of a sequence (p < ceil(local_len / P)) is numbered
 *     block_table[b][p / ppb] * ppb + p % ppb (ppb = block_size / P) and covers
 *     rows [page*P, page*P + P) of a rank's flat pool [num_blocks*block_size][576].
 *   - A (rank, sequence) cut into n splits: split s < n covers subpages
 *     [s*np/n, (s+1)*np/n) (floor) of the np subpages the longest row of the
 *     sequence needs on that rank; slots s >= n are empty ([np, np)). n = NS
 *     unless wave balancing (dims.base_splits) chooses fewer.
 *
 * Conventions shared by every call:
 *   - Every pointer argument named as device memory must point to device memory
 *     of the current device; the caller allocates and frees all buffers. The
 *     library never allocates, frees, synchronises, or reads device data on the
 *     host, so every call may be captured in a CUDA graph.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   - Ranks: a call handles ranks [rank_begin, rank_begin + num_ranks) of the
 *     dcp group. One rank per call is the per-device form; all dcp ranks in one
 *     call run them as virtual shards of one device's memory.
 *   - Return value: host-checkable argument errors return DCP_ERR_INVALID_ARG or
 *     DCP_ERR_UNSUPPORTED before anything is launched; a failed launch returns
 *     DCP_ERR_CUDA. dcp_last_error() then holds a message (thread-local).
 *   - Data errors found on the device never trap: the kernel ORs a
 *     DCP_STATUS_* bit into *status (a device word the caller zeroes), masks the
 *     offending work and carries on.
 *   - All integers are int32 unless stated; all arrays are dense, row-major,
 *     with the shapes given ("nr" = num_ranks, R = batch*qlen, H = num_heads,
 *     MP = dcp_mla_max_pages(dims), NS = num_splits, MB = max_blocks_per_seq).
 */
#ifndef DCP_MLA_H
#define DCP_MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DCP_MLA_QK_DIM 576 /* q/k width: 512 latent + 64 rope */
#define DCP_MLA_V_DIM 512  /* v width: the latent part of the same cache row */

struct CUstream_st;
typedef struct CUstream_st* dcp_stream_t; /* same type as cudaStream_t */

typedef enum {
  DCP_OK = 0,
  DCP_ERR_INVALID_ARG = 1, /* a size, pointer or rank range is invalid     */
  DCP_ERR_UNSUPPORTED = 2, /* valid, but outside what the kernels support  */
  DCP_ERR_CUDA = 3         /* a CUDA launch or runtime call failed         */
} dcp_status;

/* Bits ORed into the device status word. */
#define DCP_STATUS_BAD_SEQ_LEN 0x1u     /* seq_len < 0, or < qlen when causal     */
#define DCP_STATUS_LOCAL_OVER_BOUND 0x2u /* local length > max_local_len (clamped) */
#define DCP_STATUS_BAD_BLOCK_ID 0x4u    /* block id outside [0, num_blocks)        */
#define DCP_STATUS_BAD_PAGE 0x8u        /* partial kernel met an invalid page id   */
#define DCP_STATUS_TIMEOUT 0x10u        /* an on-device wait gave up (bounded)     */
#define DCP_STATUS_BAD_SPLIT 0x20u      /* split bounds outside [0, MP]            */
#define DCP_STATUS_Q_RANGE 0x40u        /* |q| > 65504: the FP8-cache path computes
                                           q.k in f16, which cannot hold it        */

typedef enum { DCP_KV_BF16 = 0, DCP_KV_FP8_E4M3 = 1 } dcp_kv_dtype;

/* Static problem description (host memory, read during the call only). For a
 * captured graph every field is fixed; the data that varies between replays
 * (seq_lens, block_table, q, kv) lives in device buffers. */
typedef struct {
  int32_t batch;              /* B sequences, >= 0 (0: every call is a no-op)  */
  int32_t qlen;               /* verify rows per sequence, >= 1                */
  int32_t num_heads;          /* H query heads, 1..1024                        */
  int32_t dcp;                /* W ranks in the dcp group, >= 1                */
  int32_t interleave;         /* S, 1 <= S <= block_size, block_size % S == 0  */
  int32_t block_size;         /* tokens per physical block on each rank        */
  int32_t max_blocks_per_seq; /* MB, block_table row stride; MB*block_size must
                                 be >= max_local_len                           */
  int32_t max_local_len;      /* static bound on every rank-local length       */
  int32_t num_blocks;         /* NB, blocks in each rank's pool                */
  int32_t num_splits;         /* NS, split slots per (rank, sequence)          */
  int32_t causal;             /* 1: per-row causal boundary; 0: whole sequence */
  int32_t base_splits;        /* 0 (or NS): every (rank, sequence) takes NS
                                 equal splits. 1..NS-1: wave balancing (see
                                 dcp_mla_metadata): each takes base_splits,
                                 and the shortest ones, whose work items would
                                 otherwise run in a part-filled last wave of the
                                 device, take more, up to NS                   */
} dcp_mla_dims;

/* Subpage size for a block size: min(128, largest power of two dividing it),
 * or -1 if block_size <= 0. ("[ROCm][MLA][DCP] Support causal multi-token
 * verification", Implementation item 2 and the review on the subpage bound.) */
int32_t dcp_mla_subpage_size(int32_t block_size);

/* MP = ceil(max_local_len / subpage), the page-table row length at the static
 * bound; -1 if the dims are invalid. */
int32_t dcp_mla_max_pages(const dcp_mla_dims* dims);

/* Validate dims and a rank range without launching anything. */
dcp_status dcp_mla_check_dims(const dcp_mla_dims* dims, int32_t rank_begin, int32_t num_ranks);

/*
 * Step 1+2: per-row rank-local lengths, subpages and split bounds.
 * Defined by: "Support Kimi-K3 DCP with DSpark" (review: local length formula);
 * "[ROCm][MLA][DCP] Support causal multi-token verification" (Implementation
 * items 1, 2 and 5); "Context Parallel Guide (PCP & DCP)" ("How it works" 1).
 *
 *   seq_lens    device int32 [B]           global lengths (incl. verify tokens)
 *   block_table device int32 [B][MB]       shared block ids; entries past the
 *                                          ones a sequence needs are not read
 *   row_len     device int32 [nr][R]       out: rank-local length of each row
 *                                          (row = b*qlen + j), clamped to
 *                                          max_local_len
 *   page_ids    device int32 [nr][B][MP]   out: subpage ids, -1 past the last
 *                                          needed subpage or for a bad block id
 *   split_beg,  device int32 [nr][B][NS]   out: subpage range of each split
 *   split_end
 *   status      device uint32 [1]          in/out: DCP_STATUS_BAD_SEQ_LEN,
 *                                          _LOCAL_OVER_BOUND, _BAD_BLOCK_ID ORed
 * Every output element is written (bit-exact, padding included).
 *
 * Wave balancing (0 < dims.base_splits < NS): the partial kernel runs C work
 * items at once (C = dcp_mla_concurrent_items()). With every (rank, sequence)
 * of the whole dcp group cut into base_splits, N = live * row_tiles * base_splits
 * items (live: pairs with a non-empty longest row; row_tiles =
 * ceil(qlen*H/128)). If the last wave is at most half full (0 < N mod C <= C/2),
 * the u = ceil((N mod C) / (row_tiles*base_splits)) shortest live pairs (ties:
 * the later pair, in rank-major order, is shorter) share the C slots of that wave:
 * pair j of them takes base_splits*k splits, k = floor(C / (u*row_tiles*
 * base_splits)) plus one for the first (C - that*u*row_tiles*base_splits) /
 * (row_tiles*base_splits) of them, at most NS, at most one split per 8 tiles of
 * 64 tokens, never fewer than base_splits. The choice depends on seq_lens and the
 * dims only, never on rank_begin/num_ranks, so a per-rank call cuts exactly as
 * the call for the whole group does.
 */
dcp_status dcp_mla_metadata(const dcp_mla_dims* dims, const int32_t* seq_lens,
                            const int32_t* block_table, int32_t rank_begin, int32_t num_ranks,
                            int32_t* row_len, int32_t* page_ids, int32_t* split_beg,
                            int32_t* split_end, uint32_t* status, dcp_stream_t stream);

/* Work items (clusters of two CTAs) of dcp_mla_partial that the current device
 * runs at once; -1 if there is no device or the query fails (dcp_last_error()
 * then says why). Host only. */
int32_t dcp_mla_concurrent_items(void);

/*
 * Step 3: split-KV absorbed-MLA partial attention on each rank's local KV.
 * Defined by: "[ROCm][MLA][DCP] Support causal multi-token verification",
 * Implementation item 3 (unreduced partial outputs with base-2 statistics);
 * "Context Parallel Guide (PCP & DCP)", "Decode" (each rank attends its 1/dcp
 * of the KV) and "How it works" 4 (FP8 with a per-tensor scale).
 *
 *   q           device bf16 [R][H][576]     query rows (row = b*qlen + j)
 *   kv          device [nr][NB][block_size][576], E4M3 codes (uint8) or bf16;
 *               the pool of rank rank_begin+k starts at element k*NB*bs*576
 *   kv_scale    device float [1]: per-tensor dequantisation scale (NULL = 1)
 *   softmax_scale  multiplies q.k (e.g. 1/sqrt(192))
 *   row_len, page_ids, split_beg, split_end: dcp_mla_metadata's outputs for the
 *               same dims and ranks
 *   part_o      device float [nr][NS][R][H][512]  out: per-split normalised
 *               output sum_t 2^(s_t - m) v_t / l   (0 for an empty split; not
 *               written for a slot s >= 1 with split_beg == split_end, whose m
 *               is -inf: readers skip the output of every -inf split)
 *   part_m      device float [nr][NS][R][H]  out: m = max_t s_t, where
 *               s_t = softmax_scale * kv_scale * log2(e) * (q . k_t) (base 2);
 *               -inf for an empty split
 *   part_l      device float [nr][NS][R][H]  out: l = sum_t 2^(s_t - m)
 *   workspace   device, 16-byte aligned, dcp_mla_workspace_size(dims, num_ranks)
 *               bytes, or NULL. The call first orders the work items (rank,
 *               sequence, split, 128-row tile) by tile count, longest first, so
 *               that items of very different lengths finish together, and drops
 *               the items of empty slots s >= 1 (the item of slot 0 writes their
 *               m and l). Up to 65536 items; beyond that, and with NULL, every
 *               item runs, in natural order. part_m, part_l and every part_o that
 *               readers use are bit-identical either way.
 *   status      device uint32 [1]            in/out: DCP_STATUS_BAD_PAGE,
 *               DCP_STATUS_BAD_SPLIT, DCP_STATUS_TIMEOUT, DCP_STATUS_Q_RANGE
 * Tokens at or beyond a row's length, and pages with invalid ids, never reach
 * the result (invalid ids also set DCP_STATUS_BAD_PAGE).
 */
dcp_status dcp_mla_partial(const dcp_mla_dims* dims, const void* q, const void* kv,
                           dcp_kv_dtype kv_dtype, const float* kv_scale, float softmax_scale,
                           int32_t rank_begin, int32_t num_ranks, const int32_t* row_len,
                           const int32_t* page_ids, const int32_t* split_beg,
                           const int32_t* split_end, float* part_o, float* part_m,
                           float* part_l, void* workspace, uint32_t* status,
                           dcp_stream_t stream);

/*
 * Test of the failure path of dcp_mla_partial (same arguments and checks): the
 * softmax warps withhold their arrivals on the barrier that tells the score issuer
 * the q tile is in tensor memory, so the issuer's bounded wait runs out after
 * q_wait_ns (in (0, 4e9]) instead of 4 s. Every work item then stops in order:
 * DCP_STATUS_TIMEOUT is ORed into *status, every role leaves its loop, in-flight
 * tensor-core work is drained and tensor memory freed; the partial outputs are
 * not meaningful. No wait is unbounded, nothing traps, and the context stays
 * usable for the next call.
 */
dcp_status dcp_mla_partial_hold_q(const dcp_mla_dims* dims, const void* q, const void* kv,
                                  dcp_kv_dtype kv_dtype, const float* kv_scale,
                                  float softmax_scale, int32_t rank_begin, int32_t num_ranks,
                                  const int32_t* row_len, const int32_t* page_ids,
                                  const int32_t* split_beg, const int32_t* split_end,
                                  float* part_o, float* part_m, float* part_l, void* workspace,
                                  uint32_t* status, uint64_t q_wait_ns, dcp_stream_t stream);

/* Bytes of device workspace dcp_mla_partial takes for these dims and num_ranks. */
dcp_status dcp_mla_workspace_size(const dcp_mla_dims* dims, int32_t num_ranks, size_t* bytes);

/*
 * Step 4: LSE merge of all splits of all ranks into the BF16 output.
 * Defined by: "Context Parallel Guide (PCP & DCP)", "Decode" (LSE-correct and
 * reduce the per-rank partials); "[ROCm][MLA][DCP] Support causal multi-token
 * verification", Implementation item 3 (base-2 statistics -> BF16 output plus
 * natural-log LSE).
 *
 *   part_o, part_m, part_l  dcp_mla_partial's outputs for the same ranks
 *   out       device bf16 [R][H][512]   out: sum over ranks and splits of
 *             2^(m-M) l o / sum 2^(m-M) l, rounded to nearest even (0 if empty)
 *   lse       device float [R][H]       out: natural-log LSE of the merged row,
 *             -inf if no rank has a token
 *   rank_lse  device float [nr][R][H]   out (optional, NULL to skip): each
 *             rank's own natural-log LSE, -inf for an empty rank-local row
 *   status    never written (the merge has no data-dependent failure and no
 *             wait); kept so the step's calls share one signature; may be NULL
 * With num_ranks < dcp the result merges only the given ranks.
 */
dcp_status dcp_lse_merge(const dcp_mla_dims* dims, int32_t num_ranks, const float* part_o,
                         const float* part_m, const float* part_l, void* out, float* lse,
                         float* rank_lse, uint32_t* status, dcp_stream_t stream);

/*
 * The whole verify step (metadata, partial attention and merge over all dcp
 * ranks, exactly as the three calls above with dims->num_splits) for callers
 * that cannot allocate device memory: the pages have no counterpart of this
 * call; it exists for code that must not call cudaMalloc (inside allocator
 * callbacks, or under a runtime that owns the device heap).
 *
 *   seq_lens, block_table, q, kv, kv_scale, softmax_scale: as above
 *   out  device bf16 [R][H][512], lse device float [R][H]: as dcp_lse_merge
 *   status device uint32 [1]: in/out, as above
 * Intermediates live in a fixed 32 MiB device array inside the library (held on
 * every GPU that loads it until exit); dims needing more return
 * DCP_ERR_UNSUPPORTED before any launch. The call allocates nothing. The first
 * call on a device looks up the array's device address (make that first call
 * before any stream capture on that device). Every call shares the array and it
 * keeps the last call's contents: calls that overlap on the GPU race.
 */
dcp_status dcp_mla_verify_noalloc(const dcp_mla_dims* dims, const int32_t* seq_lens,
                                  const int32_t* block_table, const void* q, const void* kv,
                                  dcp_kv_dtype kv_dtype, const float* kv_scale,
                                  float softmax_scale, void* out, float* lse, uint32_t* status,
                                  dcp_stream_t stream);

/*
 * The step before the path: writing the new (verify) tokens' latent KV rows
 * into the interleaved rank pools.
 * Defined by: "Context Parallel Guide (PCP & DCP)", "How it works" 2 (new-token
 * KV is written interleaved via slot_mapping, -1 for tokens a rank does not own)
 * and 4 (FP8 cache with one per-tensor scale); "Support Kimi-K3 DCP with DSpark"
 * (the owning rank of global position p and the slot on that rank), with the
 * interleave of the "--dcp-config" table.
 *
 * dcp_kv_slot_mapping:
 *   seq_lens     device int32 [B]      global lengths incl. the qlen new tokens;
 *                                      new token j of sequence b is at global
 *                                      position seq_lens[b] - qlen + j
 *   block_table  device int32 [B][MB]  shared block ids
 *   slot_mapping device int32 [nr][R]  out: pool row (block*block_size + offset)
 *                                      of token row b*qlen+j in the pool of rank
 *                                      rank_begin+k, or -1 where that rank does
 *                                      not own the token or the slot is invalid
 *   status       device uint32 [1]     in/out: DCP_STATUS_BAD_SEQ_LEN (seq_len <
 *                                      qlen), DCP_STATUS_LOCAL_OVER_BOUND (local
 *                                      index >= MB*block_size),
 *                                      DCP_STATUS_BAD_BLOCK_ID (id outside [0, NB))
 * dcp_kv_write:
 *   slot_mapping device int32 [nr][R]  dcp_kv_slot_mapping's output
 *   kv_new       device bf16 [R][576]  the new tokens' latent rows (row b*qlen+j)
 *   kv_scale     device float [1]      FP8 pools: code = E4M3(x / kv_scale) with
 *                                      x / kv_scale an IEEE fp32 division, rounded
 *                                      to nearest even, saturated to +-448 (NULL =
 *                                      1); ignored for BF16 pools (bits copied)
 *   pool         device [nr][NB][block_size][576] E4M3 codes or bf16: the rows
 *                named by slot_mapping are overwritten, nothing else is touched
 * Entries of slot_mapping outside [-1, NB*block_size) set DCP_STATUS_BAD_PAGE and
 * are skipped.
 */
dcp_status dcp_kv_slot_mapping(const dcp_mla_dims* dims, const int32_t* seq_lens,
                               const int32_t* block_table, int32_t rank_begin, int32_t num_ranks,
                               int32_t* slot_mapping, uint32_t* status, dcp_stream_t stream);
dcp_status dcp_kv_write(const dcp_mla_dims* dims, const int32_t* slot_mapping, const void* kv_new,
                        dcp_kv_dtype kv_dtype, const float* kv_scale, int32_t num_ranks,
                        void* pool, uint32_t* status, dcp_stream_t stream);

/*
 * The step after the path: the cross-rank exchange in the all-to-all wire
 * format, and project-before-merge.
 * Defined by: "Context Parallel Guide (PCP & DCP)", "Decode" (each rank returns
 * its output and LSE; they are LSE-corrected and summed so that every rank ends
 * with its slice of the heads), "comm_backend" (a2a: one all-to-all with the LSE
 * packed alongside the output, the fp32 LSE carried as two 16-bit halves of the
 * BF16 buffer, combine done locally) and "enable_project_before_merge" (a
 * per-head W_V applied before the merge commutes with it and shrinks the payload
 * from kv_lora_rank to v_head_dim values per head).
 *
 * Wire format. Destination rank d (of G = dims->dcp) owns heads [d*Hg, (d+1)*Hg),
 * Hg = H / G (H must be a multiple of G). The chunk a source sends to d is
 * dcp_a2a_chunk_words(dims, P) 16-bit words: [R][Hg][P] BF16 outputs (P =
 * payload: 512, or the projected width), then [R][Hg][2] LSE words (the low then
 * the high 16 bits of the float32 natural-log LSE, -inf for an empty rank), then
 * zero words up to a multiple of 8. A source's send buffer is [G][chunk]: an
 * all-to-all of equal splits delivers send_s[d] to rank d as its recv[s].
 *
 * dcp_a2a_chunk_words: words of one chunk; -1 if dims or payload are invalid.
 *
 * dcp_a2a_pack: for each rank k < num_ranks of the partials (dcp_mla_partial's
 * outputs), merges its splits into its normalised output O_k (rounded to BF16,
 * nearest even) and its LSE_k, and writes them into its send buffer (P = 512).
 *   send     device, 16-byte aligned, [num_ranks][G][chunk words(512)]   out
 *   status   never written (no data-dependent failure, no wait); may be NULL
 *
 * dcp_a2a_project: project-before-merge of packed send buffers: every BF16
 * output O_k of send is projected by its head's W_V on the tensor cores (fp32
 * accumulation), and send_projected receives the projection rounded to BF16
 * (P = payload) with the same LSE words.
 *   send            device, 16-byte aligned: dcp_a2a_pack's output    in
 *   w_v             device bf16 [H][payload][512], 16-byte aligned: row p of
 *                   head h holds the 512 weights of projected value p
 *   payload         a multiple of 16 in [16, 256]
 *   send_projected  device, 16-byte aligned, [num_ranks][G][chunk words(payload)]
 *   status          device uint32 [1] or NULL: DCP_STATUS_TIMEOUT if a wait on
 *                   the tensor cores gives up (bounded)
 *
 * dcp_a2a_combine: for destination ranks dst_begin .. dst_begin+num_dst-1, the
 * combine of the G chunks each received:
 *   LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s (0 and -inf if
 *   every source is empty).
 *   recv        device, 16-byte aligned: the chunk from source s to destination
 *               dst_begin+i starts at word i*dst_stride + s*src_stride (both
 *               multiples of 8). After a real all-to-all each rank passes its own
 *               recv buffer (num_dst 1, src_stride = chunk words); with all ranks
 *               on one device the send buffers of dcp_a2a_pack serve directly
 *               (src_stride = G*chunk words, dst_stride = chunk words).
 *   out         device bf16 [R][H][payload]: the destinations' heads are written
 *   lse         device float [R][H]: the destinations' heads are written
 *   status      never written (no data-dependent failure, no wait); may be NULL
 */
int64_t dcp_a2a_chunk_words(const dcp_mla_dims* dims, int32_t payload);

/*
 * Step 3 and the pack of the exchange in one call, for one split: the partial
 * attention of dcp_mla_partial, with each rank's normalised output rounded to BF16
 * (nearest even) and its natural-log LSE written straight into its all-to-all send
 * buffer, in the wire format of dcp_a2a_pack (P = 512), instead of the fp32 partials.
 * Defined by: "[ROCm][MLA][DCP] Support causal multi-token verification",
 * Implementation item 3 (each rank's partial output and LSE) and "Context Parallel
 * Guide (PCP & DCP)", comm_backend a2a (the output travels as BF16 with the fp32 LSE
 * in two 16-bit halves); a rank with one split has nothing to merge before it sends.
 *
 *   dims->num_splits must be 1 and num_heads a multiple of dcp (else
 *   DCP_ERR_UNSUPPORTED); the other arguments as for dcp_mla_partial
 *   send      device, 16-byte aligned, [num_ranks][dcp][dcp_a2a_chunk_words(dims,
 *             512)] 16-bit words, out: the same bits dcp_mla_partial followed by
 *             dcp_a2a_pack would write (a one-split LSE is (m + log2 l) ln 2)
 *   status    device uint32 [1], in/out: as for dcp_mla_partial
 */
dcp_status dcp_mla_partial_packed(const dcp_mla_dims* dims, const void* q, const void* kv,
                                  dcp_kv_dtype kv_dtype, const float* kv_scale,
                                  float softmax_scale, int32_t rank_begin, int32_t num_ranks,
                                  const int32_t* row_len, const int32_t* page_ids,
                                  const int32_t* split_beg, const int32_t* split_end,
                                  void* send, void* workspace, uint32_t* status,
                                  dcp_stream_t stream);
dcp_status dcp_a2a_pack(const dcp_mla_dims* dims, int32_t num_ranks, const float* part_o,
                        const float* part_m, const float* part_l, void* send, uint32_t* status,
                        dcp_stream_t stream);
dcp_status dcp_a2a_project(const dcp_mla_dims* dims, int32_t num_ranks, const void* send,
                           const void* w_v, int32_t payload, void* send_projected,
                           uint32_t* status, dcp_stream_t stream);
dcp_status dcp_a2a_combine(const dcp_mla_dims* dims, int32_t payload, const void* recv,
                           int64_t src_stride, int64_t dst_stride, int32_t dst_begin,
                           int32_t num_dst, void* out, float* lse, uint32_t* status,
                           dcp_stream_t stream);

/* Message for the last non-OK return on this thread ("" if none). */
const char* dcp_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DCP_MLA_H */
