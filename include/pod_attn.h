/*
 * pod_attn.h — C ABI of the GB300 (sm_103a) hybrid prefill+decode attention library.
 *
 * One launch computes, for one attention layer of one serving iteration:
 *   - the causal chunked-prefill ("extend") attention of each prompt chunk against its cached
 *     prefix plus the earlier tokens of the same chunk, and
 *   - the single-query decode attention of each decoding sequence,
 * both over one paged K/V cache (block size 16, grouped-query attention).
 *
 * Sources (web pages; titles and sections are what the citations below name):
 *   [POD]    "POD-Attention: hybrid batching" digest of the ASPLOS 2025 paper, Silicon & Systems
 *            (siliconandsystems.com/ko/articles/pod-attention-hybrid-batching).
 *   [BEYOND] "Week 6: Beyond PyTorch: Custom Kernel과 vLLM" lecture (core-sig.pytorch.kr).
 *   [LLMSO]  "LLMSO - W4 - Optimization & Frameworks" (seojhoon.tistory.com).
 *
 * What is computed (the definition every variant reaches, up to rounding order):
 *   [BEYOND] §"Attention에 적용하기": out = softmax(q·Kᵀ·scale)·V, with the causal rule of
 *   §"Non-Causal vs. Causal Attention" and the extend semantics of
 *   §"한 스텝에 여러 종류의 request 섞기": a prefill token at local index i of a chunk of q_len
 *   tokens whose sequence holds kv_len cached rows (the chunk's own K/V included) sits at
 *   absolute position p = kv_len - q_len + i and attends to rows 0..p. A decode token is an
 *   extend of one token: it attends to all kv_len rows.
 *   [POD] §"가상 CTA와 SM별 균형": fusing the two operations reorders independent tiles only,
 *   it does not change the mathematical result.
 *
 * Conventions shared by every entry point:
 *   - head_dim D is 128 or 64, the paged block size is 16 tokens, all tensors are bf16 (IEEE
 *     bfloat16, little-endian), accumulation is fp32, outputs are rounded once to bf16.
 *   - Layouts (row-major, innermost last, no padding):
 *       q_prefill, o_prefill : [num_prefill_tokens][num_q_heads][D]   (tokens of all chunks,
 *                                                                      concatenated)
 *       q_decode,  o_decode  : [num_decode_seqs][num_q_heads][D]
 *       k_pool, v_pool       : [num_blocks][num_kv_heads][16][D]      (one (block, kv-head)
 *                                                                      is 32*D bytes contiguous)
 *       block_tables         : int32 [num_prefill_seqs + num_decode_seqs][max_blocks_per_seq];
 *                              row s maps logical block j of sequence s to a physical block
 *                              ([BEYOND] §"PagedAttention", [LLMSO] §"PagedAttention —
 *                              메모리 단편화를 없애는 커널"). Prefill sequences come first, then
 *                              decode sequences. Entries at or beyond ceil(kv_len/16) are never
 *                              read.
 *       cu_seqlens_q         : int32 [num_prefill_seqs + 1], cu[0] = 0, cu[Np] =
 *                              num_prefill_tokens; chunk s owns tokens [cu[s], cu[s+1]).
 *       kv_lens              : int32 [num_prefill_seqs + num_decode_seqs], prefill sequences
 *                              first. kv_len counts cached rows including this step's new
 *                              tokens, whose K/V must already be in the pool.
 *   - Query head h reads kv-head h / (num_q_heads / num_kv_heads) ([LLMSO] §"KV 헤드 줄이기").
 *   - The caller owns every device buffer and every stream. The library owns only the opaque
 *     host plan (and the two CUDA events a plan holds), freed by pod_attn_plan_destroy.
 *   - No C++ exception crosses this boundary. Every function returns a status or a value.
 *   - pod_attn_run never allocates device memory and never synchronises the host.
 */
#ifndef POD_ATTN_H_
#define POD_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. Negative values are errors. */
typedef enum {
  POD_ATTN_OK = 0,
  POD_ATTN_ERR_INVALID_ARG = -1,  /* a null pointer, a bad length or an inconsistent shape */
  POD_ATTN_ERR_UNSUPPORTED = -2,  /* head_dim not 128 or 64, block_size != 16, group size > 8 */
  POD_ATTN_ERR_WORKSPACE = -3,    /* workspace too small or not 256-byte aligned */
  POD_ATTN_ERR_CUDA = -4,         /* a CUDA runtime call failed (no device, launch error, ...) */
  POD_ATTN_ERR_BAD_INDEX = -5,    /* device-detected: a block-table entry outside [0, num_blocks) */
  POD_ATTN_ERR_TIMEOUT = -6       /* device-detected: a bounded pipeline wait ran out */
} pod_attn_status;

/* How the plan's work is launched. All three compute identical results on identical inputs;
 * they differ only in scheduling ([POD] §"동시 실행만으로 부족한 이유" and
 * §"재현과 장비 평가 기준" compare exactly these three). */
typedef enum {
  POD_ATTN_FUSED = 0,   /* one persistent launch; each CTA picks prefill or decode work by SM */
  POD_ATTN_SERIAL = 1,  /* a prefill-only launch, then a decode-only launch, on `stream` */
  POD_ATTN_STREAMS = 2  /* prefill on `stream`, decode on `stream2`, joined back on `stream` */
} pod_attn_variant;

/* Shapes of one hybrid batch. */
typedef struct {
  int32_t num_q_heads;         /* Hq >= 1 */
  int32_t num_kv_heads;        /* Hkv >= 1, Hq % Hkv == 0, Hq / Hkv <= 8 */
  int32_t head_dim;            /* 128 or 64 */
  int32_t block_size;          /* must be 16 */
  int32_t num_prefill_seqs;    /* Np >= 0 */
  int32_t num_prefill_tokens;  /* sum of chunk lengths; 0 iff Np == 0 */
  int32_t num_decode_seqs;     /* Nd >= 0 */
  int32_t num_blocks;          /* physical blocks in each of k_pool and v_pool */
  int32_t max_blocks_per_seq;  /* row length of block_tables */
  float scale;                 /* softmax scale, finite and > 0; typically 1/sqrt(128) */
} pod_attn_problem;

/* Planner and launch options. Zero-initialise for defaults. */
typedef struct {
  int32_t num_sms;          /* SMs the planner sizes the grid for; 0 = query the current device */
  int32_t ctas_per_sm;      /* 0 or 1: one persistent CTA per SM, which holds a prefill slot and
                               a decode slot side by side and all of the SM's shared memory and
                               TMEM; larger values return POD_ATTN_ERR_UNSUPPORTED, negative
                               ones POD_ATTN_ERR_INVALID_ARG */
  int32_t max_prefill_ctas; /* cap on the CTAs that take prefill items: only CTAs 0 .. cap - 1
                               run prefill work (the others' prefill slots run decode items from
                               the start), so a long prefill cannot crowd decode work out of
                               every SM ([POD] §"가상 CTA와 SM별 균형"); the
                               planner sizes prefill splits for that many slots. 0 = every CTA;
                               values above the SM count mean every CTA; negative values return
                               POD_ATTN_ERR_INVALID_ARG */
  int32_t decode_splits;    /* force this many KV splits per decode (seq, kv-head), at most 64
                               (more are capped); 0 = auto */
  int32_t prefill_splits;   /* force this many KV splits per prefill output (128-row tile of
                               one chunk and head block), at most 8; 0 = auto */
  int32_t instrument;       /* nonzero: record (SM, kind, start, end) per work item */
  pod_attn_variant variant; /* launch variant, see above */
  int32_t non_causal;       /* nonzero: prefill chunk tokens attend to every row of their
                               sequence, later chunk tokens included ("Week 6: Beyond PyTorch:
                               Custom Kernel과 vLLM", §"Non-Causal vs. Causal Attention");
                               0 = causal (default) */
  int32_t kv_fp8;           /* nonzero: the plan is for pod_attn_run_decode_fp8 (an e4m3 cache;
                               decode work only), which runs four 4-warp decode groups per SM
                               and sizes its items for them; such a plan is rejected by the
                               bf16 entry points, and a plan without it by the FP8 one */
} pod_attn_options;

typedef struct pod_attn_plan_s* pod_attn_plan_t;

/* Summary of a plan (what the planner decided). */
typedef struct {
  int32_t num_prefill_items;  /* virtual prefill CTAs: (chunk, 128-row tile of 128/hp tokens
                                 x hp q-heads of one kv-head group, kv-split) */
  int32_t num_decode_items;   /* virtual decode CTAs: (seq, kv-head, kv-split) */
  int32_t num_units;          /* outputs assembled from more than one split */
  int32_t num_sms;            /* SM count the grid was sized for */
  int32_t ctas_per_sm;        /* 1 */
  int32_t max_prefill_ctas;   /* CTAs that take prefill items (the cap, at most num_sms) */
  int32_t grid_fused;         /* CTAs of the fused launch */
  int32_t grid_prefill;       /* CTAs of the prefill-only launch (serial / streams) */
  int32_t grid_decode;        /* CTAs of the decode-only launch (serial / streams) */
  int32_t smem_bytes;         /* dynamic shared memory per CTA (one budget for both kinds) */
  int32_t threads_per_cta;
  int32_t item_words;         /* int32 words per work item in pod_attn_plan_items' output */
  uint64_t workspace_bytes;   /* same as pod_attn_workspace_bytes */
  double est_prefill_flops;   /* algorithmic FLOPs: 4*d*Hq per visible (query, key) pair */
  double est_prefill_bytes;   /* algorithmic bytes: K/V once per kv-head, Q in, O out */
  double est_decode_bytes;    /* algorithmic bytes: every cached K/V row once, q in, o out */
  double est_decode_flops;
} pod_attn_plan_info;

/* Per-item record written when options.instrument is set ([POD] §"예측 가능한 지연시간과 진단":
 * the runtime should expose the virtual-CTA mix, occupancy and tile choice). */
typedef struct {
  int32_t smid;      /* SM that ran the item */
  int32_t kind;      /* 0 = prefill, 1 = decode */
  int32_t item;      /* index within its kind's item list */
  int32_t cta;       /* blockIdx.x of the CTA that ran it */
  uint64_t t_start;  /* %globaltimer, ns */
  uint64_t t_end;
} pod_attn_item_record;

/* Plan one hybrid batch on the host ([POD] §"가상 CTA와 SM별 균형": enumerate virtual prefill
 * and decode CTAs, limit prefill splits, size the grid by SM; §"동시 실행만으로 부족한 이유":
 * avoid wave-quantisation tails).
 *   problem         : shapes (read only).
 *   h_cu_seqlens_q  : host int32 [Np + 1] (read only, may be NULL when Np == 0).
 *   h_kv_lens       : host int32 [Np + Nd] (read only, may be NULL when Np + Nd == 0).
 *   options         : may be NULL (defaults).
 *   out             : receives a new plan, owned by the caller until pod_attn_plan_destroy.
 * Host only: it touches no device memory. With options->num_sms > 0 it calls no CUDA function
 * except cudaEventCreate (whose failure is tolerated; the STREAMS variant then reports
 * POD_ATTN_ERR_CUDA at run time).
 * Errors: INVALID_ARG (nulls, scale not finite or not > 0, kv_len < q_len, q_len < 1, decode kv_len < 1, kv_len beyond
 * max_blocks_per_seq*16, cu_seqlens not starting at 0 or not non-decreasing, token total
 * mismatch), UNSUPPORTED (head_dim, block size, group size), CUDA (num_sms == 0 and no device). */
pod_attn_status pod_attn_plan(const pod_attn_problem* problem, const int32_t* h_cu_seqlens_q,
                              const int32_t* h_kv_lens, const pod_attn_options* options,
                              pod_attn_plan_t* out);

/* Device workspace the plan needs, in bytes (0 for a NULL plan). Holds the work lists, the
 * scheduling counters, split-KV partials and the optional instrumentation records. */
size_t pod_attn_workspace_bytes(pod_attn_plan_t plan);

/* Copy the plan's work lists into the workspace and zero its counters and status word, on
 * `stream`, as one host-to-device copy of a host image the plan keeps (the work lists at their
 * workspace offsets after the zeroed control words). Asynchronous with respect to the device;
 * the host image is staged before the call returns, so the plan may be destroyed afterwards.
 * Must be called once after pod_attn_plan and before the first pod_attn_run with this
 * workspace; a workspace serves one plan at a time. Calling it again resets the device status.
 *   workspace       : device pointer, 256-byte aligned, >= pod_attn_workspace_bytes(plan).
 * Errors: INVALID_ARG (null plan/workspace), WORKSPACE (too small / misaligned), CUDA. */
pod_attn_status pod_attn_upload(pod_attn_plan_t plan, void* workspace, size_t workspace_bytes,
                                void* stream);

/* Launch the hybrid attention for the uploaded plan (asynchronous on `stream`).
 *   q_prefill, o_prefill : device bf16, see layouts (may be NULL when Np == 0).
 *   q_decode,  o_decode  : device bf16, see layouts (may be NULL when Nd == 0).
 *   k_pool, v_pool       : device bf16 paged pools, 16-byte aligned.
 *   d_block_tables       : device int32 [Np + Nd][max_blocks_per_seq].
 *   d_cu_seqlens_q, d_kv_lens : device copies of the arrays given to pod_attn_plan (same
 *                          values; the kernels read q offsets and kv lengths from them).
 *   workspace            : the workspace passed to pod_attn_upload for this plan.
 *   stream, stream2      : cudaStream_t values (NULL = legacy default stream); stream2 is
 *                          used by the STREAMS variant only and may equal NULL otherwise.
 * Inputs are read only; o_prefill / o_decode are overwritten entirely. Runs of the same
 * workspace must not overlap in time. The counters reset themselves at the end of a run, so
 * back-to-back runs need no further upload. Launch-time errors are returned here; errors the
 * kernels detect (BAD_INDEX, TIMEOUT) land in the workspace status word, see
 * pod_attn_last_device_status. */
pod_attn_status pod_attn_run(pod_attn_plan_t plan, const void* q_prefill, const void* q_decode,
                             const void* k_pool, const void* v_pool,
                             const int32_t* d_block_tables, const int32_t* d_cu_seqlens_q,
                             const int32_t* d_kv_lens, void* o_prefill, void* o_decode,
                             void* workspace, size_t workspace_bytes, void* stream,
                             void* stream2);

/* pod_attn_run with the iteration's KV append in front: the K and V rows of this iteration's new
 * tokens are written into the paged pools, then the attention reads them — the step that
 * precedes attention in a serving iteration ("Week 6: Beyond PyTorch: Custom Kernel과 vLLM",
 * §"PagedAttention": the paged cache grows by appending; §"한 스텝에 여러 종류의 request 섞기").
 *   k_new, v_new : device bf16 [T_p + Nd][Hkv][D], 16-byte aligned: row i < T_p is prefill
 *                  token i (chunks in cu_seqlens order), row T_p + d is decode sequence d's token.
 *                  Token i of chunk s is written at position kv_len[s] - q_len(s) + i of sequence
 *                  s, decode d's token at position kv_len[Np + d] - 1, through the block tables
 *                  (whose blocks for those positions must exist).
 *   k_pool, v_pool : written at exactly those rows; every other row is only read.
 * Other arguments as pod_attn_run. FUSED does the append inside its one launch (each CTA writes
 * a share, then the items that read new rows wait, bounded, until all shares are done; the
 * launch is cooperative, so all CTAs are resident); SERIAL and STREAMS run the append as a
 * launch of its own ahead of theirs. Results equal pod_attn_run on pools that already hold the
 * rows. Errors: as pod_attn_run; INVALID_ARG also for NULL or misaligned k_new / v_new; a
 * block-table entry outside the pool is reported as BAD_INDEX (the row is not written). */
pod_attn_status pod_attn_run_append(pod_attn_plan_t plan, const void* q_prefill,
                                    const void* q_decode, const void* k_new, const void* v_new,
                                    void* k_pool, void* v_pool, const int32_t* d_block_tables,
                                    const int32_t* d_cu_seqlens_q, const int32_t* d_kv_lens,
                                    void* o_prefill, void* o_decode, void* workspace,
                                    size_t workspace_bytes, void* stream, void* stream2);

/* Decode attention over an FP8 KV cache: e4m3 values (1 sign, 4 exponent bits with bias 7, 3
 * mantissa bits, no infinities) with one fp32 scale per (kv-head, channel) for K and one per
 * cached (row, kv-head) for V ([LLMSO] §"2-4. 고급 KV 캐싱 기법": per-channel scales suit K,
 * whose outliers sit in particular channels, per-token scales suit V), so the cache takes half
 * the bytes of bf16 and the decode step, which reads the whole cache ([BEYOND] §"KV Cache"),
 * about half the time. Cached K row j, channel c = e4m3(k_pool8[..][j][c]) * k_scale[g][c]; V row j,
 * channel c = e4m3(v_pool8[..][j][c]) * v_scale[..][j]. The query and output stay bf16.
 * Arithmetic: e4m3 is converted to f16 exactly; q * k_scale and the softmax weights times
 * v_scale are rounded to f16 for the tensor cores (magnitudes above 65504 saturate there);
 * scores, softmax and accumulation are fp32.
 *   plan          : a plan made with options.kv_fp8 set, no prefill sequences and head_dim 128
 *                   (else UNSUPPORTED); its variant is not used: the work runs as one launch.
 *   q_decode, o_decode : device bf16 [Nd][Hq][128], as pod_attn_run.
 *   k_pool8, v_pool8   : device uint8 [num_blocks][Hkv][16][128], 16-byte aligned.
 *   d_k_scale          : device fp32 [Hkv][128], 16-byte aligned.
 *   d_v_scale          : device fp32 [num_blocks][Hkv][16], 16-byte aligned.
 *   d_block_tables, d_kv_lens, workspace, stream : as pod_attn_run.
 * Errors: as pod_attn_run. */
pod_attn_status pod_attn_run_decode_fp8(pod_attn_plan_t plan, const void* q_decode,
                                        const void* k_pool8, const void* v_pool8,
                                        const float* d_k_scale, const float* d_v_scale,
                                        const int32_t* d_block_tables, const int32_t* d_kv_lens,
                                        void* o_decode, void* workspace, size_t workspace_bytes,
                                        void* stream);

/* The iteration's KV append for an FP8 cache: one new token per decode sequence, written at
 * position kv_len - 1 of its sequence (the plan's lengths) through the block tables, quantised to
 * e4m3 ([LLMSO] §"2-4. 고급 KV 캐싱 기법": K per channel, V per token).
 *   K row, channel c : e4m3(k / k_scale[g][c]) with the given per-(kv-head, channel) scales.
 *   V row            : scale = max over the row's channels of |v| / 448 (1 when that max is 0),
 *                      stored in v_scale at the row; values e4m3(v / scale).
 *   Divisions are IEEE binary32 (round to nearest); e4m3 codes round to nearest even and
 *   saturate at +-448.
 *   plan            : a plan made with options.kv_fp8 set (decode work only, head_dim 128), whose
 *                     work lists were uploaded to `workspace` (pod_attn_upload); else UNSUPPORTED.
 *   k_new, v_new    : device bf16 [Nd][Hkv][128], 16-byte aligned, decode d's row at index d.
 *   k_pool8, v_pool8: device uint8 [num_blocks][Hkv][16][128]; only the new rows are written.
 *   d_k_scale       : device fp32 [Hkv][128], read only.
 *   d_v_scale       : device fp32 [num_blocks][Hkv][16]; the new rows' entries are written.
 * One small launch on `stream`, ahead of pod_attn_run_decode_fp8 on the same stream. A
 * block-table entry outside the pool is reported as BAD_INDEX in the workspace status word
 * (pod_attn_last_device_status), and that row is not written. */
pod_attn_status pod_attn_append_fp8(pod_attn_plan_t plan, const void* k_new, const void* v_new,
                                    void* k_pool8, void* v_pool8, const float* d_k_scale,
                                    float* d_v_scale, const int32_t* d_block_tables,
                                    void* workspace, size_t workspace_bytes, void* stream);

/* Synchronise `stream`, read and clear the device status word of `workspace`.
 * workspace NULL reads the status word of pod_attn_run_static's scratch array on the current
 * device instead (the runs made through that entry point).
 * Returns OK, BAD_INDEX, TIMEOUT, or CUDA if the synchronisation itself failed. After
 * BAD_INDEX or TIMEOUT the outputs of that run are unspecified and the workspace must be
 * re-uploaded before the next run (pod_attn_run_static uploads on every call). */
pod_attn_status pod_attn_last_device_status(pod_attn_plan_t plan, void* workspace, void* stream);

/* Fill *info with the plan summary. Errors: INVALID_ARG. */
pod_attn_status pod_attn_get_plan_info(pod_attn_plan_t plan, pod_attn_plan_info* info);

/* Resource features of a plan and their buckets. No counterpart in code on the pages: the
 * "POD-Attention" digest (§"스케줄링 입력으로 쓰는 자원 특성") proposes describing prefill chunks
 * and decode groups by CTA count, shared memory, arithmetic intensity and bytes read, in coarse
 * buckets, so that the kernel can publish a few validated (bucket, latency) pairs from which an
 * outer scheduler chooses (e.g. the largest prefill chunk whose measured tail latency fits a
 * token-to-token budget, §"예측 가능한 지연시간과 진단"). Host only, integer arithmetic: equal
 * batches give equal buckets, bit for bit. */
typedef struct {
  int64_t prefill_flops;     /* 4*D*Hq per visible (query, key) pair of the prefill chunks */
  int64_t read_bytes;        /* algorithmic bytes: each sequence's K/V rows once per kv-head
                                (4*D B per row and kv-head), q in and o out (4*D B per token and
                                q-head) */
  int32_t prefill_ctas;      /* virtual prefill CTAs (work items) */
  int32_t decode_ctas;       /* virtual decode CTAs */
  int32_t grid;              /* hardware CTAs of the fused launch */
  int32_t smem_per_cta;      /* dynamic shared memory of one CTA, bytes */
  int32_t tmem_cols_per_cta; /* TMEM columns one CTA allocates (0: decode-only plan) */
  int32_t bucket_flops;      /* 0 without prefill, else bit length of ceil(prefill_flops / 2^30) */
  int32_t bucket_bytes;      /* 0 without work, else bit length of ceil(read_bytes / 2^20) */
  int32_t bucket_ctas;       /* bit length of prefill_ctas + decode_ctas */
  double intensity;          /* prefill_flops / read_bytes (FLOP per byte) */
} pod_attn_bucket;

/* Fill `out` for `plan`. Errors: INVALID_ARG (null plan or out). */
pod_attn_status pod_attn_plan_bucket(pod_attn_plan_t plan, pod_attn_bucket* out);

/* Copy the host work lists: prefill items first, then decode items, then the unit table, each
 * item info.item_words (8) int32 words: kind (0 prefill, 1 decode); prefill chunk index or
 * decode sequence index; prefill tile index (chunk tokens 128/hp * t ..) or decode kv-head;
 * prefill first query head
 * (decode 0); first key row of the split; one past its last key row; the unit index of a split
 * output (-1 when the item writes its output directly); the split's index within the unit. A
 * unit is 4 words: split count, first partial slot, kind, 0.
 *   out   : host buffer of `capacity` int32 words, or NULL to query the size only.
 *   count : receives the number of words (written, or needed when out is NULL).
 * Used to check the planner bit for bit. Errors: INVALID_ARG (null plan/count, capacity too
 * small). */
pod_attn_status pod_attn_plan_items(pod_attn_plan_t plan, int32_t* out, size_t capacity,
                                    size_t* count);

/* Copy the instrumentation records of the last run (synchronises `stream`).
 *   out    : host array of `capacity` records; count receives the number written (one per
 *            item, prefill items first). Errors: INVALID_ARG (instrumentation off), CUDA. */
pod_attn_status pod_attn_read_records(pod_attn_plan_t plan, const void* workspace,
                                      pod_attn_item_record* out, size_t capacity,
                                      size_t* count, void* stream);

/* Allocation-free launch of the FUSED variant. The pages have no counterpart to this entry
 * point; it exists for callers that cannot call cudaMalloc to obtain a workspace: for example a
 * plugin running inside a host program whose device memory belongs to that program's own
 * allocator (the plugin has no way to ask it for memory, and a private cudaMalloc would compete
 * with it or fail once the program has reserved the device), or a latency-critical loop that
 * cannot afford cudaMalloc's implicit device synchronisation.
 *
 * Instead of a caller workspace it uses one library-owned scratch array of
 * POD_ATTN_STATIC_SCRATCH_BYTES bytes, a file-scope __device__ array: every GPU that loads the
 * library holds it until the process exits. Each call copies the plan's work lists into that
 * array and clears its status word, scheduling counters and merge counters (on `stream`), then
 * launches the fused kernel exactly as pod_attn_run does. It calls no cudaMalloc, cudaFree or
 * other allocating routine.
 *   plan            : a plan made with variant POD_ATTN_FUSED and without instrumentation; its
 *                     pod_attn_workspace_bytes must not exceed POD_ATTN_STATIC_SCRATCH_BYTES.
 *   stream          : a stream of the current device (the array used is the current device's).
 *   other arguments : as for pod_attn_run (inputs read only, outputs overwritten).
 * The first call on a device looks up the array's device address on that device (with the
 * device current); make that first call before any stream capture on the device.
 * All calls share the one array, which keeps the last call's contents: calls whose work
 * overlaps on the GPU (different streams, or another host thread) race and give wrong results;
 * serialise them. Device-detected errors (bad block index, timeout) are recorded in the
 * array's status word: read them with pod_attn_last_device_status(plan, NULL, stream).
 * Errors: INVALID_ARG (null plan, variant other than FUSED, an instrumented plan, a stream of
 * another device, null/misaligned tensors), UNSUPPORTED (a plan for the e4m3 cache), WORKSPACE
 * (plan needs more than POD_ATTN_STATIC_SCRATCH_BYTES), CUDA. */
#define POD_ATTN_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)
pod_attn_status pod_attn_run_static(pod_attn_plan_t plan, const void* q_prefill,
                                    const void* q_decode, const void* k_pool,
                                    const void* v_pool, const int32_t* d_block_tables,
                                    const int32_t* d_cu_seqlens_q, const int32_t* d_kv_lens,
                                    void* o_prefill, void* o_decode, void* stream);

/* Free the plan (NULL is ignored). */
void pod_attn_plan_destroy(pod_attn_plan_t plan);

/* Static English description of a status code. */
const char* pod_attn_status_string(pod_attn_status status);

/* Test hook for the bounded-wait failure path (no GPU fault involved): launches one CTA whose
 * thread 0 waits on an mbarrier nobody arrives on, for at most `timeout_us` microseconds, and
 * records POD_ATTN_ERR_TIMEOUT in the workspace status word when the limit runs out (the same
 * bounded wait every pipeline wait of the attention kernels uses, there with a 4 s limit).
 *   workspace : device pointer with at least 256 bytes, its first 8 bytes zeroed by the caller
 *               (pod_attn_upload does this for a plan's workspace).
 * Read the outcome with pod_attn_last_device_status. Errors: INVALID_ARG, CUDA. */
pod_attn_status pod_attn_selftest_timeout(void* workspace, int32_t timeout_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* POD_ATTN_H_ */
