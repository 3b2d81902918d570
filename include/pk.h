/*
 * pk.h -- C ABI of the packed mixed-mask variable-length attention library
 * for GB300 (sm_103a).
 *
 * The operation ("[RFC]: HunyuanImage 3.0 deployment", Proposed Change, P0
 * "Packed Attention for Multi-Request Batching"): requests of different
 * resolutions are packed back to back into one token stream described by
 * cu_seqlens, with no padding and no explicit (bsz,1,seqlen,seqlen) mask
 * (Motivation, item (1)).  Each packed sequence carries the model's
 * generalized causal mask (same page, P0 "Attention mask challenge";
 * "Model structure", item 1):
 *
 *   query i of a sequence sees key j of the same sequence iff
 *     j <= i, or i lies in an IMAGE segment and j lies in that same segment.
 *
 * Nothing attends across sequences.  Query head h reads key/value head
 * h / (hq / hkv) (grouped-query attention, contiguous groups).
 *
 *   out[t,h,:] = sum_j softmax_j(scale * q[t,h,:].k[j,g,:]) v[j,g,:]
 *   lse[h,t]   = ln sum_j exp(scale * q[t,h,:].k[j,g,:])   (visible j only)
 *
 * Tensors (all caller-owned device memory, bf16 = IEEE bfloat16):
 *   q   [Tq][hq][d]  bf16, rows contiguous, 16-byte aligned base
 *   k,v [Tk][hkv][d] bf16, rows contiguous, 16-byte aligned base
 *   out [Tq][hq][d]  bf16, written for every query row
 *   lse [hq][Tq]     fp32, natural log, written for every query row
 * With pk_plan_create, Tq = Tk = cu_seqlens[num_seqs].  With
 * pk_plan_create_layout, Tq = cu_seqlens_q[num_seqs] and Tk = num_kv_rows.
 * A query row that sees no key of its key range (possible only when the
 * range starts after position 0) gets out = 0 and lse = -inf.
 *
 * Ownership: the library never allocates device memory.  A plan owns host
 * memory only; its device image lives in a caller-allocated buffer of
 * pk_plan_device_bytes() bytes that must outlive every launch using it.
 * Each launch also takes a caller-allocated workspace of
 * pk_attn_workspace_bytes() bytes (an fp16 copy of the values, see
 * pk_attn_fwd).
 * Thread safety: a plan is read-only after pk_plan_upload; concurrent
 * launches on one plan are safe when each has its own workspace.
 */
#ifndef PK_H_
#define PK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream (identical to cudaStream_t / CUstream). */
typedef struct CUstream_st* pk_stream_t;

typedef enum pk_status {
  PK_OK = 0,
  PK_ERR_INVALID_ARG = 1,   /* malformed descriptors, null pointer, bad size */
  PK_ERR_UNSUPPORTED = 2,   /* head_dim not in {64, 128}, device not sm_103 */
  PK_ERR_ALIGNMENT = 3,     /* a tensor base is not 16-byte aligned */
  PK_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
  PK_ERR_TIMEOUT = 5,       /* device: a bounded wait ran out (in dev_status) */
  PK_ERR_DEVICE_CHECK = 6,  /* device: an internal consistency check failed */
  PK_ERR_NOT_UPLOADED = 7,  /* plan has no device image yet */
  PK_ERR_OUT_OF_MEMORY = 8, /* a host memory allocation failed */
  PK_ERR_RANGE = 9,         /* device: a value of magnitude >= 2^16 (outside fp16) */
  PK_ERR_TOO_LARGE = 10     /* the plan needs more than pk_attn_fwd_noalloc's static scratch */
} pk_status;

typedef enum pk_seg_type { PK_TEXT = 0, PK_IMAGE = 1 } pk_seg_type;

/* One segment of a sequence: tokens [start, start+len) of the packed stream
 * (global token index), all TEXT or all IMAGE.  Adjacent IMAGE segments are
 * distinct images: neither sees the other's later tokens. */
typedef struct pk_segment {
  int32_t start;
  int32_t len;
  int32_t type;
} pk_segment;

/* A segment in its sequence's own position space: positions [start,
 * start+len) of sequence `seq`, all TEXT or all IMAGE. */
typedef struct pk_seq_segment {
  int32_t seq;
  int32_t start;
  int32_t len;
  int32_t type;
} pk_seq_segment;

/*
 * General layout ("[RFC]: HunyuanImage 3.0 deployment", Proposed Change, P0
 * "KV Cache Transfer Integration for DiT": the text prefix's keys/values come
 * from the AR stage, so the queries of a step are a subset of positions of
 * the sequence; and the page-table keys of the recipe's paged-KV mode).
 * Sequence s covers positions [0, L_s), tiled by its segments (segs ordered
 * by seq, then start).  Its queries are the packed rows
 * [cu_seqlens_q[s], cu_seqlens_q[s+1]) at positions q_pos0[s] + i; its keys
 * are positions k_pos0[s] + j, j < cu_seqlens_k[s+1] - cu_seqlens_k[s],
 * stored at row cu_seqlens_k[s] + j of k/v (block_table == NULL), or at row
 * block_table[s * blocks_per_seq + p / 128] * 128 + p % 128 for position p
 * (paged: 128-row blocks, k_pos0[s] a multiple of 128, num_kv_rows the pool
 * rows, a multiple of 128).  q_pos0 / k_pos0 may be NULL (all zero).  The
 * mask is the one of the whole sequence.  All pointers are host memory.
 */
typedef struct pk_layout {
  int32_t num_seqs;
  const int32_t* cu_seqlens_q;
  const int32_t* q_pos0;
  const int32_t* cu_seqlens_k;
  const int32_t* k_pos0;
  const pk_seq_segment* segs;
  int32_t num_segs;
  const int32_t* block_table;
  int32_t blocks_per_seq;
  int32_t num_kv_rows;
} pk_layout;

typedef struct pk_plan pk_plan;

/* Summary of a plan (host data, for callers and tests). */
typedef struct pk_plan_info {
  int32_t total_tokens;     /* T */
  int32_t num_seqs;
  int32_t hq, hkv, head_dim;
  int32_t num_items;        /* work items: (q-tile, kv head, query-head pair) */
  int32_t num_ctas;         /* persistent CTAs launched by pk_attn_fwd */
  int32_t num_full_tiles;   /* (item, k-tile) visits with no mask math */
  int32_t num_partial_tiles;/* (item, k-tile) visits with per-element mask */
  int32_t kv_rows;          /* Tk: rows of the key/value tensors */
  int64_t visible_pairs;    /* per query head, over the whole pack */
  double useful_flops;      /* 4 * d per visible pair and query head of the
                               plan's items (4 * d * hq * visible_pairs
                               unless the plan is a shard) */
} pk_plan_info;

/* Device work item, 32 bytes, as stored in the plan image (exposed for
 * tests and tools).  A work item is one 128-row query tile of one sequence
 * for up to two query heads of the same key/value head. */
typedef struct pk_work_item {
  int32_t q_start;   /* global token index of the tile's first query row */
  int32_t q_rows;    /* valid query rows in the tile, 1..128 */
  int32_t kv_start;  /* contiguous keys: row of the key range's first key;
                        paged: index of its first block in the block table */
  int32_t n_kt;      /* 128-key tiles visited, from kv_start upwards */
  int32_t n_full;    /* leading tiles visible to every valid row (no mask) */
  int32_t hq0;       /* query head of slot 0 */
  int32_t hq1;       /* query head of slot 1, or -1 when the slot is empty */
  int32_t hkv;       /* key/value head shared by both slots */
} pk_work_item;

/*
 * Build a plan (host only, no device work).
 *   cu_seqlens : host int32[num_seqs+1]; cu_seqlens[0] == 0, non-decreasing.
 *                Empty sequences are allowed and produce no work.
 *   segs       : host pk_segment[num_segs], in token order, non-empty, tiling
 *                every sequence exactly (no segment crosses a sequence end).
 *   hq, hkv    : query / key-value heads, hq % hkv == 0.
 *   head_dim   : 64 or 128 (else PK_ERR_UNSUPPORTED).
 *   num_ctas   : persistent CTAs to schedule for; 0 = the current device's
 *                SM count (needs a CUDA device).
 * On success *out owns a new plan (free with pk_plan_destroy).  On failure
 * *out is set to NULL and a status is returned.
 */
pk_status pk_plan_create(const int32_t* cu_seqlens, int32_t num_seqs,
                         const pk_segment* segs, int32_t num_segs, int32_t hq,
                         int32_t hkv, int32_t head_dim, int32_t num_ctas,
                         pk_plan** out);

/* Same planner for a general layout (see pk_layout); head_dim and num_ctas
 * as for pk_plan_create.  Keys may be paged only with head_dim 64 or 128 and
 * 128-row blocks. */
pk_status pk_plan_create_layout(const pk_layout* layout, int32_t hq, int32_t hkv,
                                int32_t head_dim, int32_t num_ctas, pk_plan** out);

/*
 * One rank's share of a plan, for running one pack on several GPUs without
 * an exchange (the pages' CFG-parallel and head-split schemes,
 * "Parallelism Acceleration Guide").  The plan's work units, one (sequence,
 * key/value head) pair each, go to ranks longest first, each to the
 * least-loaded rank; every rank computes the same assignment, so the shares
 * of ranks 0..num_ranks-1 partition the plan's work items exactly.  The
 * shard keeps its units' items, scheduled over num_ctas CTAs (0 = the
 * current device's SM count).  It is launched like any plan, on the full
 * q, k, v tensors, and writes out and lse only for its units' rows and
 * query heads; the union of the ranks' outputs is the full plan's output.
 * pk_plan_useful_flops and pk_plan_get_info's num_items and tile counts
 * describe the shard's own work.  *out owns a new plan (pk_plan_destroy).
 */
pk_status pk_plan_shard(const pk_plan* full, int32_t rank, int32_t num_ranks, int32_t num_ctas,
                        pk_plan** out);

/*
 * SM-pair kernel, opt-in (head_dim 128, pk_attn_fwd and the calls built on
 * it; the FP8 entries keep the one-CTA kernel).  With enable != 0 the
 * attention runs on clusters of two CTAs on SM pairs: each pair computes
 * its two query tiles as M = 256 tensor-core products (tcgen05 cta_group::2),
 * each SM holding half of every key and value tile, so each SM copies half
 * the key/value bytes per tile.  Results are bit-identical to the one-CTA
 * kernel.  The plan pairs, one query head at a time, query tiles that
 * read the same key/value tiles (same first key row, key/value head and
 * query head) by their key-tile count; a pair visits the larger count (the
 * other rows see the extra tiles fully masked).  Measured on GB300 against
 * the one-CTA kernel: faster on packs of long sequences (+3 to +4% on the
 * two 24,832-token sequences of the high-res edit pack), slower on packs of
 * short ones (-2% on the mixed-resolution pack, -6 to -15% on the CFG
 * pair); the default head-pair clusters (pk_plan_set_kv_share) are faster
 * than it on every pack measured, so it is off by default.  The pages have
 * no counterpart; it is a tuning option of this library.
 *   PK_ERR_INVALID_ARG for a null plan; PK_ERR_UNSUPPORTED when enabling a
 *   plan that has no pair schedule (head_dim other than 128, or built for
 *   fewer than two CTAs).  Takes effect at the next launch; not thread-safe
 *   against launches running on the plan.
 */
pk_status pk_plan_set_sm_pairs(pk_plan* plan, int32_t enable);

/*
 * Head-pair clusters, on by default at head_dim 128 where the plan has
 * their schedule (an even number of query heads per key/value head: every
 * work item then holds two query heads); available, off by default, at
 * head_dim 64, where they measured 1.7% slower than one CTA per SM.  A cluster of two CTAs on
 * neighbouring SMs runs each of its items with one query head per CTA; the
 * two stream the same key and value tiles, and each CTA copies half of
 * every tile from global memory into the shared memory of both (TMA
 * multicast within the cluster), so the pack's keys and values leave L2
 * half as often.  Each CTA computes exactly what the one-CTA kernel computes
 * for its head: results are bit-identical with the schedule on or off.
 * Applies to pk_attn_fwd and the calls built on it, and to
 * pk_attn_fwd_fp8; pk_plan_set_sm_pairs takes precedence, and
 * pk_attn_fwd_fp8_pv keeps the one-CTA kernel.  Measured on GB300: +1 to
 * +8% on the d = 128 packs.  The pages have no counterpart; it is a
 * tuning option of this library.  enable = 0 selects the one-CTA kernel.
 *   PK_ERR_INVALID_ARG for a null plan; PK_ERR_UNSUPPORTED when enabling a
 *   plan without the schedule.  Takes effect at the next launch; not
 *   thread-safe against launches running on the plan.
 */
pk_status pk_plan_set_kv_share(pk_plan* plan, int32_t enable);

/* 1 when launches of the plan run on head-pair clusters (their schedule
 * exists and pk_plan_set_kv_share has them on; pk_plan_set_sm_pairs still
 * takes precedence), else 0 (also for a null plan). */
int32_t pk_plan_kv_share(const pk_plan* plan);

/* Bytes of the device image of the plan (work list, per-CTA offsets, the
 * per-row key limit and, for paged keys, the block table). */
size_t pk_plan_device_bytes(const pk_plan* plan);

/* Copy the plan's device image into dev_buf (caller-owned, >= 256-byte
 * aligned, >= pk_plan_device_bytes bytes) on `stream`, and remember dev_buf.
 * Asynchronous: the plan's host memory stays valid until destroy. */
pk_status pk_plan_upload(pk_plan* plan, void* dev_buf, size_t bytes,
                         pk_stream_t stream);

/* Bytes of the workspace a launch with `plan` needs: Tk * hkv * head_dim * 2
 * (the fp16 copy of the value rows). */
size_t pk_attn_workspace_bytes(const pk_plan* plan);

/* Bytes of the workspace pk_attn_fwd_fp8_pv needs with `plan`: the
 * transposed E4M3 copy of the value rows, hkv * head_dim bytes per row, each
 * sequence's key rows rounded up to a multiple of 16 (contiguous keys) or
 * the pool's rows rounded up to 16 (paged keys).  0 for a null plan. */
size_t pk_attn_workspace_bytes_fp8_pv(const pk_plan* plan);

/*
 * Launch the attention forward on `stream` (asynchronous): two kernels, the
 * conversion of the value rows the plan reads from bf16 to fp16 into the
 * workspace, then the attention (on head-pair clusters when
 * pk_plan_kv_share(plan) is 1, one CTA per SM otherwise).
 *   q, k, v   : device bf16 tensors as described above.
 *   out, lse  : device outputs as described above.
 *   scale     : softmax scale, finite and > 0 (usually 1/sqrt(head_dim)).
 *   workspace : caller-owned device memory of at least
 *               pk_attn_workspace_bytes(plan) bytes, 16-byte aligned; it
 *               receives the fp16 values at the rows of v, and must not be
 *               used by another launch until this one is done.  It may be v
 *               itself when the caller no longer needs v: the conversion is
 *               then in place and leaves fp16 values in v.
 *   dev_status: nullable device int32; on a device-side failure the kernels
 *               write PK_ERR_TIMEOUT / PK_ERR_DEVICE_CHECK there, and
 *               PK_ERR_RANGE when a value's magnitude is 2^16 or more (the
 *               caller zeroes it; it is never cleared by the library).
 * P enters the P V product in fp16 (11 significant bits), with v converted
 * to fp16 to match: exact for 2^-14 <= |v| < 2^16, rounded to fp16
 * subnormals below (absolute error at most 2^-25), saturated to 65504 (and
 * PK_ERR_RANGE reported) at 2^16 and above.  O is divided by the fp32 sum of
 * the unrounded probabilities, which also gives the LSE.
 * Argument and launch errors are returned synchronously.  Requires a device
 * of compute capability 10.3 (GB300); PK_ERR_UNSUPPORTED also if the
 * library's kernel was compiled with fewer registers per thread than its
 * warp roles share out (a build-configuration error, checked once).
 */
pk_status pk_attn_fwd(const pk_plan* plan, const void* q, const void* k,
                      const void* v, void* out, float* lse, float scale,
                      void* workspace, size_t workspace_bytes,
                      pk_stream_t stream, int32_t* dev_status);

/*
 * The two launches of pk_attn_fwd as separate calls, for callers that reuse
 * converted values (for example the text prefix's values handed over from
 * the autoregressive stage, unchanged across denoising steps) or time the
 * kernels apart.  pk_attn_convert_values writes the fp16 copy of the value
 * rows the plan reads into `workspace` (arguments, in-place use and
 * PK_ERR_RANGE as for pk_attn_fwd); pk_attn_fwd_converted runs the attention
 * on such a copy, v16 (pk_attn_workspace_bytes(plan) bytes, 16-byte
 * aligned), which it only reads.  Both asynchronous on `stream`.
 */
pk_status pk_attn_convert_values(const pk_plan* plan, const void* v, void* workspace,
                                 size_t workspace_bytes, pk_stream_t stream,
                                 int32_t* dev_status);
pk_status pk_attn_fwd_converted(const pk_plan* plan, const void* q, const void* k,
                                const void* v16, void* out, float* lse, float scale,
                                pk_stream_t stream, int32_t* dev_status);

/*
 * pk_attn_fwd for callers that cannot allocate device memory where they make
 * the call: code embedded in a host framework that owns all device memory
 * through its own pool and forbids other allocations, or a latency-critical
 * loop that must not make a call that can synchronise the device
 * (cudaMalloc and cudaFree can).  It takes no workspace: the fp16 copy of the
 * values lives in a static device array of the library, 64 MiB (67108864
 * bytes), which every device that loads the library holds until the process
 * exits.  The pages have no counterpart; it is an addition of this library.
 *   Arguments, layouts, results and dev_status as for pk_attn_fwd.
 *   PK_ERR_TOO_LARGE, before any device work, when pk_attn_workspace_bytes(plan)
 *   exceeds 64 MiB (for example 32768 key rows x 8 heads x 128 dims).
 * Every call shares the one array and leaves its contents behind; each call
 * rewrites (or zeroes) every part of it that its kernels read, so nothing
 * depends on an earlier call.  Calls that overlap on the GPU (launched on
 * different streams without ordering) race on the array: order them.  The
 * entry point's first call on a device takes the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  It allocates no memory (no cudaMalloc,
 * cudaFree or allocating library routine).
 */
pk_status pk_attn_fwd_noalloc(const pk_plan* plan, const void* q, const void* k,
                              const void* v, void* out, float* lse, float scale,
                              pk_stream_t stream, int32_t* dev_status);

/*
 * FP8 variant: queries and keys as FP8 E4M3 codes (1 sign, 4 exponent bits
 * with bias 7, 3 mantissa bits; the OCP 8-bit format), one dequantisation
 * scale each, values bf16.  The scores are scale * q_scale * k_scale *
 * (q8 . k8), computed on the tensor cores in FP8 with fp32 accumulation;
 * softmax, P V, workspace, out and lse as for pk_attn_fwd.
 *   q8 [Tq][hq][128], k8 [Tk][hkv][128] uint8 codes, 16-byte aligned;
 *   q_scale, k_scale: finite and > 0.
 * head_dim must be 128 (else PK_ERR_UNSUPPORTED).  The pages quantise their
 * linear layers to FP8 ("HunyuanImage-3.0-Instruct ...", FP8 checkpoints;
 * "MiniMax H3-Image on Vera Rubin", MXFP8 GEMMs); this is the attention of
 * such a model with FP8 queries and keys.
 */
pk_status pk_attn_fwd_fp8(const pk_plan* plan, const void* q8, float q_scale, const void* k8,
                          float k_scale, const void* v, void* out, float* lse, float scale,
                          void* workspace, size_t workspace_bytes, pk_stream_t stream,
                          int32_t* dev_status);

/*
 * All-FP8 variant: queries, keys and values as FP8 E4M3 codes, one
 * dequantisation scale each.  Scores as in pk_attn_fwd_fp8; the softmax
 * weights p (in (0, 256], relative to a running row maximum) are rounded to
 * E4M3 and the product P V runs on the tensor cores in FP8 with fp32
 * accumulation; out = v_scale * (P v8) / l with l the fp32 sum of the
 * unrounded weights, lse as for pk_attn_fwd.  The E4M3 weights carry 3
 * mantissa bits, so out is less accurate than pk_attn_fwd_fp8's (the tests
 * record the measured error); lse is unaffected.
 *   q8 [Tq][hq][128], k8 and v8 [Tk][hkv][128] uint8 codes, 16-byte aligned;
 *   q_scale, k_scale, v_scale: finite and > 0.
 *   workspace: >= pk_attn_workspace_bytes_fp8_pv(plan) bytes, 16-byte
 *   aligned; a kernel before the attention writes the transposed copy of
 *   v8 into it (keys along rows, rows 16-key aligned per sequence), which
 *   the FP8 P V product reads.
 * head_dim must be 128 (else PK_ERR_UNSUPPORTED).  Otherwise as
 * pk_attn_fwd_fp8 (dev_status, out and lse, errors).  The pages run
 * attention at FP8 on the linear layers' side only; E4M3 values and
 * weights are an addition of this library.
 */
pk_status pk_attn_fwd_fp8_pv(const pk_plan* plan, const void* q8, float q_scale, const void* k8,
                             float k_scale, const void* v8, float v_scale, void* out, float* lse,
                             float scale, void* workspace, size_t workspace_bytes,
                             pk_stream_t stream, int32_t* dev_status);

/*
 * End-to-end variant for callers holding host buffers: copies q, k, v from
 * host memory into the caller's device buffers, runs pk_attn_fwd, and copies
 * out and lse back into host memory, all on `stream` (asynchronous; pinned
 * host memory makes the copies truly asynchronous).  Device buffers are the
 * caller's (same shapes as pk_attn_fwd); v_dev also serves as the workspace
 * (its values are converted to fp16 in place).  Host buffers must stay
 * valid until the stream reaches the end of this call's work.
 */
pk_status pk_attn_fwd_host(const pk_plan* plan, const void* q_host,
                           const void* k_host, const void* v_host,
                           void* out_host, float* lse_host, void* q_dev,
                           void* k_dev, void* v_dev, void* out_dev,
                           float* lse_dev, float scale, pk_stream_t stream,
                           int32_t* dev_status);

/*
 * Host-buffer pipeline: successive steps whose inputs and outputs live in
 * host memory (pinned memory makes the copies asynchronous).  Each step's
 * host -> device copy of q, k, v, its pk_attn_fwd and its device -> host
 * copy of out and lse run on three streams of the pipeline, ordered by
 * events, so one step's copies overlap the neighbouring steps' kernels.
 * Device memory is the caller's: num_slots (1..8) sets of buffers of the
 * pk_attn_fwd shapes for `plan`, used round robin (a slot's v is its
 * launch's workspace, converted to fp16 in place); a slot is refilled only
 * after its previous kernel has read it and its previous outputs are out.
 * The pipeline creates and owns its streams and events, no device memory.
 */
typedef struct pk_dev_slot {
  void* q;
  void* k;
  void* v;
  void* out;
  float* lse;
} pk_dev_slot;

typedef struct pk_pipeline pk_pipeline;

/* slots: host array of num_slots descriptors (copied).  The plan must stay
 * alive and uploaded while the pipeline is used. */
pk_status pk_pipeline_create(const pk_plan* plan, const pk_dev_slot* slots, int32_t num_slots,
                             pk_pipeline** out);
/* Enqueue one step (asynchronous).  The host buffers must stay valid and
 * unmodified until pk_pipeline_sync returns (or the step's copy-out stream
 * has passed it). */
pk_status pk_pipeline_submit(pk_pipeline* pipe, const void* q_host, const void* k_host,
                             const void* v_host, void* out_host, float* lse_host, float scale,
                             int32_t* dev_status);
/* Wait for every submitted step. */
pk_status pk_pipeline_sync(pk_pipeline* pipe);
/* The pipeline's streams: 0 copy-in, 1 compute, 2 copy-out (NULL otherwise). */
pk_stream_t pk_pipeline_stream(const pk_pipeline* pipe, int32_t which);
/* Waits for outstanding work, then frees the streams and events. */
void pk_pipeline_destroy(pk_pipeline* pipe);

void pk_plan_destroy(pk_plan* plan);

const char* pk_status_string(pk_status status);

/* 4 * head_dim per visible (query, key) pair and query head of the plan's
 * work items: 4 * head_dim * hq * (visible pairs per head) for a whole pack,
 * the shard's part for pk_plan_shard. */
double pk_plan_useful_flops(const pk_plan* plan);

pk_status pk_plan_get_info(const pk_plan* plan, pk_plan_info* info);

/* Host copies of plan internals, for tests: the per-row key limit (index of
 * the last visible key within the row's key range, -1 for none; int32[Tq])
 * and the CTA-ordered work list (pk_work_item[num_items]) with per-CTA
 * offsets (int32[num_ctas+1]). */
pk_status pk_plan_get_kv_limit(const pk_plan* plan, int32_t* out, int64_t n);
pk_status pk_plan_get_items(const pk_plan* plan, pk_work_item* items,
                            int64_t n_items, int32_t* cta_offsets,
                            int64_t n_offsets);
/* The SM-pair schedule (pk_plan_set_sm_pairs), for tests: *num_pairs and
 * *num_clusters (0 when the plan has none); with non-null arrays of at
 * least 2 * num_pairs items and num_clusters + 1 offsets, the
 * cluster-ordered (rank 0, rank 1) item pairs and the per-cluster offsets
 * in pairs.  PK_ERR_INVALID_ARG for a null plan or short arrays. */
pk_status pk_plan_get_pairs(const pk_plan* plan, int32_t* num_pairs, int32_t* num_clusters,
                            pk_work_item* items, int64_t n_items, int32_t* cluster_offsets,
                            int64_t n_offsets);

/* The head-pair cluster schedule (pk_plan_set_kv_share), for tests:
 * *num_clusters (0 when the plan has none, whether enabled or not); with
 * non-null arrays of at least pk_plan_info.num_items items and
 * num_clusters + 1 offsets, the cluster-ordered items and the per-cluster
 * offsets.  PK_ERR_INVALID_ARG for a null plan or short arrays. */
pk_status pk_plan_get_share(const pk_plan* plan, int32_t* num_clusters, pk_work_item* items,
                            int64_t n_items, int32_t* cluster_offsets, int64_t n_offsets);

/* Element types of pk_lse_merge's tensors. */
typedef enum pk_dtype { PK_DTYPE_BF16 = 0, PK_DTYPE_F32 = 1 } pk_dtype;

/* One partial attention result: o [T][H][d] (dtype) and its natural-log LSE
 * lse [H][T] fp32, both device memory, as written by pk_attn_fwd over one
 * block of keys. */
typedef struct pk_merge_part {
  const void* o;
  const float* lse;
  int32_t dtype;
} pk_merge_part;

/*
 * Merge partial attentions over disjoint key sets into the attention over
 * their union ("Parallelism Acceleration Guide", Ring Attention: each ring
 * step's block result is folded into the running output):
 *   lse[h,t]   = ln sum_c exp(lse_c[h,t])
 *   out[t,h,:] = sum_c exp(lse_c[h,t] - lse[h,t]) * o_c[t,h,:]
 * A part with lse_c = -inf adds nothing (its o_c is not read); a row with no
 * finite lse_c gets out = 0 and lse = -inf; a NaN lse_c gives NaN.  LSE
 * inputs must be finite or -inf.
 *   parts     : host array of num_parts (1..16) descriptors.
 *   T, H, d   : rows, heads, head dim; d in {8, 16, 32, 64, 128, 256}.
 *   out       : device [T][H][d] of out_dtype; lse_out device fp32 [H][T].
 * out may be the o of a part of the same dtype and lse_out the lse of a
 * part (in-place accumulation); no other overlap is allowed.  o and out
 * 16-byte aligned, LSEs 4-byte aligned.  Asynchronous on `stream`.
 * dev_status: nullable device int32 that receives PK_ERR_TIMEOUT if one of
 * the kernel's bounded waits runs out (as for pk_attn_fwd).
 */
pk_status pk_lse_merge(const pk_merge_part* parts, int32_t num_parts, int32_t T, int32_t H,
                       int32_t d, void* out, int32_t out_dtype, float* lse_out,
                       pk_stream_t stream, int32_t* dev_status);

/* Upper bound of every device-side wait, in nanoseconds (default 4e9).
 * Process-wide; applies to launches made after the call. */
void pk_set_wait_timeout_ns(uint64_t ns);

/* Self-test of the bounded wait: launches one CTA that waits on a barrier
 * nothing arrives at, for at most `timeout_ns`, and writes PK_ERR_TIMEOUT to
 * dev_status when the wait runs out. */
pk_status pk_debug_wait_timeout(int32_t* dev_status, uint64_t timeout_ns,
                                pk_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PK_H_ */
