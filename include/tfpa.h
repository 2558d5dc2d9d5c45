/*
 * tfpa: GQA attention over a paged KV cache, for GB300 (sm_103a).
 *
 * Keys and values live in 256-position pages drawn from one shared pool; a
 * stream reaches its pages through its own page table (TensorFold PR #2011,
 * "What this changes": every stream takes 256-position pages from the core
 * pool).  A stream may instead hold a contiguous slab; both are read with one
 * arithmetic, so a stream's output is the same bytes paged or not, batched or
 * alone (PR #1373, "What changes"; Issue #1344, "Conclusion").
 *
 * Layouts (all row-major, element = bf16 or one e4m3 byte):
 *   pool  K, V : [num_pages][hkv][256][128]   key j of kv head g of a paged
 *                stream is pool[PT[j/256]][g][j%256]  (PR #2011, review
 *                "Is paged output the same as windowed output?": base
 *                PT[k0/256]*PS + (hk*256 + k0%256)*D)
 *   slab  K, V : [hkv][slab_cap][128]          key j of kv head g is slab[g][j]
 *   q, out     : bf16 [rows][hq][128]
 *   k_rows, v_rows (KV write input): bf16 [rows][hkv][128]
 *   lse        : float [rows][hq], natural log, nullable
 * Query head h reads kv head h / (hq/hkv).
 *
 * Rows and segments.  A call covers `rows` query rows; row r belongs to
 * segment row_seg[r] (an index into `segs`) and sits at cache position
 * row_pos[r]; it attends to keys 0..row_pos[r] of its segment (causal).
 * Rows of one segment should be contiguous with consecutive positions (a
 * decode/verify group or a prompt chunk); other orders are accepted and run
 * as more, smaller groups.
 *
 * Memory and ownership.  Every buffer is allocated by the caller.  Pointers
 * marked DEVICE are device memory of the current device; HOST arrays are read
 * during the call only and not retained.  The library allocates no device
 * memory, keeps no state between calls except host-side caches (TMA tensor
 * maps, per host thread; each device's SM count) and the plans a caller
 * creates (a plan may own a CUDA graph, see tfpa_plan_capture), and never
 * synchronises the stream: all work is enqueued on `stream`.
 *
 * Pinned host memory on the decode path.  Where DEVICE is marked below for
 * q, k_rows, v_rows, out or lse of tfpa_decode, tfpa_decode_tree,
 * tfpa_decode_append, tfpa_merge, tfpa_write_kv and tfpa_write_kv_rope (and
 * their plans), and for a device-mode plan's buffer, page-locked host memory
 * mapped at its own address (cudaHostAlloc / cudaMallocHost under unified
 * addressing, or cudaHostRegister with cudaHostRegisterMapped) may stand in:
 * the kernels read and write it with plain loads and stores over the host
 * link (NVLink-C2C on a Grace-Blackwell node), with no copy-engine copy.
 * Data the host writes there before it enqueues a call is what the call
 * reads; results are the host's once the stream has passed the call.  A
 * slice with rows for the tensor-core verify path and tfpa_prefill load q
 * by TMA from device memory only: host memory there returns TFPA_EINVAL.
 * Memory that is not page-locked is not supported (and not checked).
 *
 * Threads.  Calls may be made from several host threads at once, on any
 * streams and devices: each thread builds its launch parameters in its own
 * buffers and no call takes a lock on that path (the pool ledger and the
 * static-scratch address lookup lock their own state).  Work enqueued on
 * different streams runs concurrently on the GPU, so two calls must not
 * write the same output, scratch or cache rows at once.
 * tfpa_set_launch_hook must not run while another call is in progress.
 *
 * Errors.  Every call returns TFPA_OK (0) or a negative code below and
 * enqueues nothing on error.  Kernels never trap: a page id outside
 * [0, num_pages) found on the device is skipped (its keys take no part in
 * attention; the KV write skips its rows) and sets bit 1 of cache->err_flag
 * (if non-NULL); a wait inside a kernel that gives up sets bit 2.
 */
#ifndef TFPA_H
#define TFPA_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TFPA_PAGE 256          /* positions per page (compile-time constant) */
#define TFPA_HEAD_DIM 128      /* the only head size built                  */
#define TFPA_MAX_SPLITS 32     /* split-K partials per (row, head), at most */

enum {
  TFPA_OK = 0,
  TFPA_EINVAL = -1,      /* bad dims, dtype, NULL pointer, misalignment, or a
                            softmax_scale that is not finite and positive   */
  TFPA_ERANGE = -2,      /* a position, segment or (host-mirrored) page id out of range */
  TFPA_ECAPACITY = -3,   /* scratch too small for the requested rows/splits */
  TFPA_ECUDA = -4,       /* a CUDA runtime/driver call or a launch failed    */
  TFPA_EDEVICE = -5,     /* current device is not sm_100-family (tcgen05)    */
  TFPA_ELANEMEM = -6     /* the page pool cannot hold the claim now: wait     */
};

typedef enum { TFPA_BF16 = 0, TFPA_FP8_E4M3 = 1 } tfpa_kv_dtype;

/* One stream (a segment of the call). */
typedef struct {
  int32_t seq_len;                /* valid keys, >= 1 (includes rows written by this round) */
  const int32_t* page_table;      /* DEVICE int32[ceil(seq_len/256)]; NULL => slab stream   */
  const int32_t* page_table_host; /* optional HOST mirror, checked against num_pages        */
  void* k_slab;                   /* DEVICE [hkv][slab_cap][128], slab streams only          */
  void* v_slab;
  int32_t slab_cap;               /* slab capacity in positions, multiple of 256            */
} tfpa_seg;

/* One layer's KV cache. */
typedef struct {
  tfpa_kv_dtype dtype;
  int32_t hq, hkv, head_dim;      /* hq % hkv == 0, head_dim == 128                        */
  void* k_pool;                   /* DEVICE [num_pages][hkv][256][128], 1024-byte aligned;  */
  void* v_pool;                   /*   may be NULL when no segment is paged                 */
  int32_t num_pages;
  const float* k_scale;           /* DEVICE float[hkv], fp8 only: value = e4m3 * scale      */
  const float* v_scale;
  int32_t* err_flag;              /* optional DEVICE int32: OR-ed with 1 on a bad page id,
                                     4 on a rotary position outside the table */
} tfpa_cache;

/* Split-K scratch for decode partials (float32).
 *   part_o  : DEVICE [cap_rows][hq][max_splits][128]  unnormalised outputs o
 *   part_ml : DEVICE [cap_rows][hq][max_splits][2]    (m, l): running max of the
 *             scores in log2 units (score * log2(e)) and the sum of 2^(s2 - m)
 *   arrive  : optional DEVICE uint32[cap_rows][hq], all zero before the first
 *             call.  With it, tfpa_decode merges a slice inside the partial
 *             kernel when each of its streams has at most 4 splits
 *             (seq_len <= 1,024): the last CTA to finish a split of a group
 *             of query vectors (counted here) merges that group's splits in
 *             split order, with the merge kernel's arithmetic, so the output
 *             bytes are those of the separate merge; a launch leaves every
 *             counter at zero again.  Longer streams, tfpa_decode_tree,
 *             plans in device mode and slices with rows for the tensor-core
 *             verify path keep the separate merge (a group's in-kernel merge
 *             runs on one SM at the kernel's tail: for 32 splits it was
 *             measured slower than the separate launch).  After a call that
 *             set the cache's err_flag the counters may be left non-zero:
 *             zero them before the next call.  NULL: always the separate
 *             merge. */
typedef struct {
  float* part_o;
  float* part_ml;
  int32_t cap_rows;               /* rows one partial launch can hold                      */
  int32_t max_splits;             /* >= tfpa_num_splits(seq_len) of every segment used     */
  uint32_t* arrive;
} tfpa_scratch;

/* KV write with rotary position embedding: tfpa_write_kv, with each row's K
 * rotated before it is stored.  The pages list "rope stores" among the paged
 * KV store's checks (PR #1373 review) without defining the rotation; this
 * reading is used: for i < 64, with c = rope_cos[t][i], s = rope_sin[t][i]
 * and t the row's rotary position,
 *   k'[i] = k[i] c - k[i+64] s,   k'[i+64] = k[i+64] c + k[i] s,
 * each product, difference and sum rounded to float32 (no fused multiply-
 * add), then stored as bf16 (round to nearest even) or as tfpa_write_kv
 * stores an fp8 value.  V is stored as tfpa_write_kv stores it.
 *   rope_pos : DEVICE int32[rows], 4-byte aligned, each in [0, rope_n); or
 *              NULL: the storage positions row_pos (then checked on the host,
 *              TFPA_ERANGE).  A device position outside the table leaves the
 *              row unwritten and ORs 4 into cache->err_flag.  The rotary
 *              position may differ from the storage position (a draft-tree
 *              node is rotated by its depth and stored at its index).
 *   rope_cos, rope_sin : DEVICE float32 [rope_n][64], 16-byte aligned.
 * Sliced like the rows.  TFPA_EINVAL for a NULL or misaligned table. */
int tfpa_write_kv_rope(const tfpa_cache* cache, const tfpa_seg* segs, int32_t nseg,
                       const void* k_rows, const void* v_rows, const int32_t* row_seg,
                       const int32_t* row_pos, const int32_t* rope_pos, const float* rope_cos,
                       const float* rope_sin, int32_t rope_n, int32_t rows,
                       cudaStream_t stream);

/* Keep: copy stored K/V rows (every kv head, the stored bytes unchanged)
 * from position keep_src[i] to keep_dst[i] of segment keep_seg[i] (HOST
 * int32[n] each), e.g. to move a draft tree's accepted path to the committed
 * positions.  The pages list "keep" among the paged store's checks (PR #1373
 * review); reading used: every source row is read before any destination is
 * written, so chains of moves within one call are exact.  Positions must lie
 * in [0, seq_len) (TFPA_ERANGE); a destination may appear only once per
 * segment (TFPA_EINVAL); at most 256 pairs a call (TFPA_ECAPACITY).  A page
 * id out of range skips that pair and ORs 1 into cache->err_flag. */
int tfpa_keep_kv(const tfpa_cache* cache, const tfpa_seg* segs, int32_t nseg,
                 const int32_t* keep_seg, const int32_t* keep_src, const int32_t* keep_dst,
                 int32_t n, cudaStream_t stream);

/* ---- Page pool admission (host) ------------------------------------------
 * The pages' memory admission (PR #2011 review, "Memory admission"): a
 * request claims its pages (prompt, max_tokens and one more forward) up front
 * when it is seated, never grows them, waits with LaneMemory when the pool is
 * full, and is turned away by fits() when it could never fit.  Reading used:
 * a claim is all or nothing and takes the lowest free page ids (pages need not
 * be contiguous, so only the free count decides); a released page may be
 * claimed again.  Thread-safe.  No CUDA call. */
typedef struct tfpa_pool tfpa_pool;
tfpa_pool* tfpa_pool_create(int32_t num_pages);      /* NULL if num_pages < 1       */
void tfpa_pool_destroy(tfpa_pool* pool);
int32_t tfpa_pool_free(const tfpa_pool* pool);        /* pages free now              */
int tfpa_pool_fits(const tfpa_pool* pool, int32_t npages);  /* 1 if npages <= pool size */
/* Claims npages pages into pages_out (HOST int32[npages], ascending).
 * TFPA_ELANEMEM when fewer are free now (nothing claimed), TFPA_ECAPACITY
 * when the pool could never hold them, TFPA_EINVAL for npages < 0 or NULL. */
int tfpa_pool_claim(tfpa_pool* pool, int32_t npages, int32_t* pages_out);
/* Returns pages (HOST int32[n]).  TFPA_EINVAL (and nothing released) if one
 * is out of range, not claimed, or listed twice. */
int tfpa_pool_release(tfpa_pool* pool, const int32_t* pages, int32_t n);

/* Device-side page-table staging (the pages stage a prompt chunk's page ids
 * between chunks, PR #2011 review, and measure host gaps from it): writes
 * pages[0..n) (HOST int32) into page_table (DEVICE int32) at [first, first+n)
 * on the stream.  The ids travel in kernel parameters (up to 2,048 a launch),
 * so there is no copy call and no host synchronisation; later work on the
 * stream sees the entries.  TFPA_EINVAL for NULL, first < 0 or n < 0. */
int tfpa_stage_pages(int32_t* page_table, int32_t first, const int32_t* pages, int32_t n,
                     cudaStream_t stream);

/* ---- Save and restore a stream's stored rows ------------------------------
 * Page-granular save/restore of a stream's K and V (PR #2011 review: save
 * and restore copies, one copy per page, and a kernel writing mapped host
 * memory measured faster than copies at 32k).  Positions [p0, p1) of segment
 * seg, every kv head, the stored bytes unchanged, to or from an image laid out
 * [K, V][hkv][p1 - p0][128] elements of the cache's dtype (2 or 1 bytes):
 *   image : a pointer the GPU can access, 16-byte aligned: pinned (page-
 *           locked) host memory, registered host memory, or device memory.
 * One kernel launch; the copy runs on the stream (no host synchronisation).
 * A page id out of range skips its rows and ORs 1 into cache->err_flag.
 * TFPA_ERANGE unless 0 <= p0 <= p1 <= seq_len; TFPA_EINVAL for a NULL or
 * misaligned image. */
int tfpa_save_kv(const tfpa_cache* cache, const tfpa_seg* seg, int32_t p0, int32_t p1,
                 void* image, cudaStream_t stream);
int tfpa_restore_kv(const tfpa_cache* cache, const tfpa_seg* seg, int32_t p0, int32_t p1,
                    const void* image, cudaStream_t stream);

/* Split policy, a function of a stream's own length only (so a stream's
 * partials never depend on its batch): pages_per_split = 1 for npages <= 16,
 * else max(2, ceil(npages / 32)); nsplit = ceil(npages / pages_per_split). */
int32_t tfpa_pages_per_split(int32_t seq_len);
int32_t tfpa_num_splits(int32_t seq_len);

/* The split count of each row as tfpa_decode_partial leaves its partials
 * (the nsplit to pass to tfpa_merge for the same rows).  Rows are grouped
 * into runs (consecutive rows of one segment at consecutive positions); a
 * run of at least 49 query vectors per kv head (ceil(nrows * G / 16) >= 4,
 * G = hq / hkv <= 128) takes the tensor-core verify path, whose splits are
 * at least 24 pages and at most 7 a stream; every other row has
 * tfpa_num_splits(seq_len).  Host only (no GPU work): nsplit is HOST
 * int32[rows].  TFPA_EINVAL / TFPA_ERANGE as tfpa_decode. */
int tfpa_row_splits(const tfpa_cache* cache, const tfpa_seg* segs, int32_t nseg,
                    const int32_t* row_seg, const int32_t* row_pos, int32_t rows,
                    int32_t* nsplit);

/* KV write (the KV store kernels that write a stream's page run, PR #1373,
 * "What changes"): row r's K and V for every kv head go to position
 * row_pos[r] of segment row_seg[r], through its page table or slab.  bf16
 * caches copy the bits; fp8 caches store e4m3(RNE, saturating) of
 * float32(x) / scale[g].  row_seg/row_pos are HOST int32[rows]. */
int tfpa_write_kv(const tfpa_cache* cache, const tfpa_seg* segs, int32_t nseg,
                  const void* k_rows, const void* v_rows,
                  const int32_t* row_seg, const int32_t* row_pos, int32_t rows,
                  cudaStream_t stream);

/* Decode/verify split-K partials (Issue #1344, "Mechanism": the partial
 * kernels write pm/pl/po, then attn_merge).  For each row r < rows, head h
 * and split s < nsplit[r]: (m, l, o) at scratch row r, where nsplit[r] is
 * what tfpa_row_splits gives for the same rows (tfpa_num_splits(seq_len),
 * or fewer for rows of a run on the tensor-core verify path).
 * Requires rows <= scratch->cap_rows (TFPA_ECAPACITY otherwise). */
int tfpa_decode_partial(const tfpa_cache* cache, const tfpa_seg* segs, int32_t nseg,
                        const void* q, const int32_t* row_seg, const int32_t* row_pos,
                        int32_t rows, float softmax_scale, const tfpa_scratch* scratch,
                        cudaStream_t stream);

/* Log-sum-exp merge of scratch rows 0..rows-1 (PR #1355: one merge per slice
 * of at most most_verify rows): out = sum_s o_s 2^(m_s-M) / sum_s l_s 2^(m_s-M),
 * lse = ln2 * (M + log2 sum_s l_s 2^(m_s-M)).  nsplit is HOST int32[rows]. */
int tfpa_merge(const tfpa_scratch* scratch, int32_t hq, int32_t rows,
               const int32_t* nsplit, void* out, float* lse, cudaStream_t stream);

/* Decode/verify attention: partial + merge, in slices of at most
 * scratch->cap_rows rows on shifted q/row-table/out pointers (PR #1355,
 * "Follow-up checks": slices never overrun the partial scratch). */
int tfpa_decode(const tfpa_cache* cache, const tfpa_seg* segs, int32_t nseg,
                const void* q, const int32_t* row_seg, const int32_t* row_pos,
                int32_t rows, float softmax_scale, const tfpa_scratch* scratch,
                void* out, float* lse, cudaStream_t stream);

/* A decode step in one call: the rows' K and V are stored (as tfpa_write_kv
 * stores them; k_rows, v_rows: DEVICE bf16 [rows][hkv][128], 16-byte
 * aligned) and the rows are decoded (as tfpa_decode decodes them), so the
 * cache and the output hold the bytes of tfpa_write_kv followed by
 * tfpa_decode.  When every run goes to the decode partial kernel and no
 * segment has two runs in the call, that kernel stores the rows itself:
 * the CTAs whose keys include a new row store it before they read it, and
 * no write launch runs.  Otherwise one KV write launch precedes the decode
 * launches.  TFPA_EINVAL for NULL or misaligned rows. */
int tfpa_decode_append(const tfpa_cache* cache, const tfpa_seg* segs, int32_t nseg,
                       const void* k_rows, const void* v_rows, const void* q,
                       const int32_t* row_seg, const int32_t* row_pos, int32_t rows,
                       float softmax_scale, const tfpa_scratch* scratch, void* out, float* lse,
                       cudaStream_t stream);

/* Draft-tree verify: tfpa_decode whose rows see the keys their ancestor
 * masks allow instead of every earlier key.  The pages' partial and merge
 * kernels index the queries, the row tables, the ancestor table (rowanc),
 * the partials and the output by row, and a sliced launch shifts the
 * ancestor table with the other row tables (PR #1355, "Follow-up checks");
 * the pages do not spell out the table's format, and this reading is used:
 *   row_anc : DEVICE uint64[rows], 8-byte aligned, read from the launch's
 *             stream.  Bit d of row_anc[r] set: the key at position
 *             row_pos[r] - d is visible to row r.  Keys more than 63
 *             positions back are always visible, keys after row_pos[r] never.
 *             Bit 0 (the row's own key) must be set.  All bits set is the
 *             causal row, and then the result equals tfpa_decode's bytes.
 * A draft tree of at most 64 nodes laid out at consecutive positions sets,
 * for node i, the bits of its ancestors and itself and every bit that
 * reaches before the root (the committed prefix).  Errors as tfpa_decode;
 * TFPA_EINVAL also for a NULL or misaligned row_anc. */
int tfpa_decode_tree(const tfpa_cache* cache, const tfpa_seg* segs, int32_t nseg,
                     const void* q, const int32_t* row_seg, const int32_t* row_pos,
                     const uint64_t* row_anc, int32_t rows, float softmax_scale,
                     const tfpa_scratch* scratch, void* out, float* lse, cudaStream_t stream);

/* Decode/verify attention for callers that cannot allocate device memory.
 *
 * Some callers cannot call cudaMalloc: code that runs inside another
 * framework's memory manager, a plug-in that may not grow its host process's
 * device footprint, or a runtime whose allocations are all made before it
 * starts serving.  This entry point needs no caller scratch: the split-K
 * partials live in one array compiled into the library (a file-scope
 * __device__ array of TFPA_STATIC_SCRATCH_SLOTS slots of 130 floats, about
 * 4.3 MB), which every device that loads the library holds until the process
 * exits.  None of the TensorFold sources has a counterpart to this entry
 * point.
 *
 * Same arguments and result as tfpa_decode without `scratch`; rows are
 * processed in slices of TFPA_STATIC_SCRATCH_SLOTS / (hq * TFPA_MAX_SPLITS)
 * rows (8 at hq = 32), which gives the same bytes as tfpa_decode.  Head
 * counts with hq * TFPA_MAX_SPLITS > TFPA_STATIC_SCRATCH_SLOTS (hq > 256) are
 * refused with TFPA_ECAPACITY.  It allocates no device memory and calls no
 * allocating CUDA or library routine.
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture.  The address is kept per device context:
 * if the context is replaced (cudaDeviceReset, then new work), the next call
 * looks it up again, so it is also a set-up call.  Every call shares the one array and it
 * keeps the last call's contents; nothing in it needs to start at zero, as
 * every slot the merge reads is written by the partial kernel of the same
 * call.  Calls that overlap on the GPU (other streams, other host threads)
 * race on the array: serialise them. */
#define TFPA_STATIC_SCRATCH_SLOTS 8192
int tfpa_decode_static(const tfpa_cache* cache, const tfpa_seg* segs, int32_t nseg,
                       const void* q, const int32_t* row_seg, const int32_t* row_pos,
                       int32_t rows, float softmax_scale, void* out, float* lse,
                       cudaStream_t stream);

/* ---- Plans: planning a call apart from enqueueing it -----------------------
 * A decode loop's host work (checks, grouping rows into runs, split counts,
 * per-CTA item ranges, tensor maps) does not need the GPU.  A plan does that
 * work for a tfpa_write_kv, tfpa_decode or tfpa_decode_append call (same
 * arguments, without the stream) and keeps the resulting launches by value; tfpa_plan_launch then
 * only enqueues them.  A loop can plan step i + 1 while the GPU runs step i,
 * so that between the host's wait for step i's output and step i + 1's
 * kernels there are only the launches.  None of the TensorFold sources has a
 * counterpart to this.
 *
 * A plan keeps the pointers it was given (device buffers, the cache's pools,
 * scales and page tables, the scratch) and reads them when its launches
 * run: they must stay valid and hold that step's data then.  Host arrays
 * (segs, row tables, host page-table mirrors) are read during the planning
 * call only.  Planning calls append to the plan in order; tfpa_plan_launch
 * enqueues every launch on `stream` in that order and may be called any
 * number of times.  A planning call that fails returns its error code (as
 * the direct call would) and leaves the plan as it was.  A plan is used by
 * one host thread at a time.  tfpa_plan_create returns NULL if host memory
 * runs out; tfpa_plan_launch returns TFPA_ECUDA if a launch fails (launches
 * before it stay enqueued). */
typedef struct tfpa_plan tfpa_plan;
tfpa_plan* tfpa_plan_create(void);
void tfpa_plan_destroy(tfpa_plan* plan);
void tfpa_plan_clear(tfpa_plan* plan);                 /* drops every planned launch */
int32_t tfpa_plan_launches(const tfpa_plan* plan);     /* launches planned so far    */
int tfpa_plan_write_kv(tfpa_plan* plan, const tfpa_cache* cache, const tfpa_seg* segs,
                       int32_t nseg, const void* k_rows, const void* v_rows,
                       const int32_t* row_seg, const int32_t* row_pos, int32_t rows);
int tfpa_plan_decode(tfpa_plan* plan, const tfpa_cache* cache, const tfpa_seg* segs,
                     int32_t nseg, const void* q, const int32_t* row_seg,
                     const int32_t* row_pos, int32_t rows, float softmax_scale,
                     const tfpa_scratch* scratch, void* out, float* lse);
int tfpa_plan_decode_append(tfpa_plan* plan, const tfpa_cache* cache, const tfpa_seg* segs,
                            int32_t nseg, const void* k_rows, const void* v_rows, const void* q,
                            const int32_t* row_seg, const int32_t* row_pos, int32_t rows,
                            float softmax_scale, const tfpa_scratch* scratch, void* out,
                            float* lse);
int tfpa_plan_launch(const tfpa_plan* plan, cudaStream_t stream);

/* Device mode: replaying a captured plan as the streams grow.
 * A plan's launches normally carry everything by value, so a CUDA graph
 * captured from tfpa_plan_launch repeats the lengths it was captured with.
 * In device mode each write, decode and merge launch instead reads the data
 * that changes as streams grow (run lengths and positions, split counts,
 * work-item and per-CTA ranges) from its own slot of a DEVICE buffer that
 * the caller owns, and the launch shapes stop depending on the lengths: a
 * decode partial launch takes one CTA per SM (at most 256) whatever its
 * work.  A decode loop then captures once [copy of the packed data into the
 * buffer, tfpa_plan_launch] and, each step, re-plans with the new lengths,
 * packs and replays.
 *
 * tfpa_plan_set_device(plan, dyn, bytes): dyn = DEVICE buffer, 16-byte
 *   aligned, `bytes` long, or NULL to go back to parameter mode.  dyn may
 *   be mapped pinned host memory (see "Pinned host memory" above): then
 *   tfpa_plan_dyn_pack may write the packed data into dyn itself, with no
 *   copy, while no launch that reads it is pending.  Only on an
 *   empty plan (after create or clear), else TFPA_EINVAL.  The plan keeps the
 *   pointer; tfpa_plan_clear keeps the mode.  A planning call whose slots do
 *   not fit returns TFPA_ECAPACITY; rows that would take the tensor-core
 *   verify path (a stream with 4 or more 16-vector m-tiles, whose grid
 *   follows the lengths) return TFPA_EINVAL.
 * tfpa_plan_dyn_bytes: bytes of the buffer the planned launches use (about
 *   4 KB per decode launch, 2.6 KB per write, 2 KB per merge).
 * tfpa_plan_dyn_pack(plan, host, bytes): writes those bytes, the data of
 *   the launches as planned now, to HOST memory `host` (the caller copies
 *   them to `dyn` before the launches run, e.g. with a copy captured in the
 *   same graph from pinned memory; the host buffer must not change while
 *   such a copy is pending).  TFPA_EINVAL outside device mode,
 *   TFPA_ECAPACITY if bytes < tfpa_plan_dyn_bytes.
 * tfpa_plan_shape: a 64-bit hash of everything the launches take by value
 *   except that data (kinds, grids, pointers, tensor maps, head counts).
 *   Two plans with the same shape may replay one captured graph; a
 *   different shape (new rows, a stream moved between pool and slab, a
 *   slice boundary moved) needs a new capture. */
int tfpa_plan_set_device(tfpa_plan* plan, void* dyn, size_t bytes);
size_t tfpa_plan_dyn_bytes(const tfpa_plan* plan);
int tfpa_plan_dyn_pack(const tfpa_plan* plan, void* host, size_t bytes);
uint64_t tfpa_plan_shape(const tfpa_plan* plan);

/* A plan as one CUDA graph, owned by the plan.
 * tfpa_plan_capture(plan, before, nbefore, after, nafter, stream) captures,
 *   on `stream` (a created stream: not NULL, not cudaStreamLegacy; nothing
 *   else may be enqueued on it meanwhile), the copies `before` (each a
 *   cudaMemcpyAsync of `bytes` from src to dst, kind inferred: e.g. a step's
 *   inputs and, in device mode, its packed data from pinned host memory),
 *   the plan's launches and the copies `after` (e.g. the output to pinned
 *   host memory), instantiates the graph and keeps it with the plan's shape
 *   (tfpa_plan_shape), replacing an earlier one.  The copies read and write
 *   their buffers when the graph runs.  TFPA_EINVAL for an empty plan, bad
 *   copies or stream; TFPA_ECUDA if capture or instantiation fails (the
 *   plan keeps its earlier graph).  Launch the plan once before its first
 *   capture on a device, so that kernel attributes are set outside capture.
 * tfpa_plan_replay(plan, stream): launches the graph on `stream`.
 *   TFPA_EINVAL if nothing was captured or the plan's shape has changed
 *   since (re-planned with other rows, streams or pointers: capture again).
 *   In device mode a loop re-plans each step (tfpa_plan_clear + planning
 *   calls), packs into the host buffer the graph's first copy reads, and
 *   replays.  The graph is destroyed with the plan; tfpa_plan_clear keeps it. */
typedef struct {
  void* dst;
  const void* src;
  size_t bytes;
} tfpa_copy;
int tfpa_plan_capture(tfpa_plan* plan, const tfpa_copy* before, int32_t nbefore,
                      const tfpa_copy* after, int32_t nafter, cudaStream_t stream);
int tfpa_plan_replay(const tfpa_plan* plan, cudaStream_t stream);

/* Causal prompt-chunk attention over the paged prefix, one pass with online
 * softmax on tcgen05/TMEM tiles (PR #2011, "hpattn_p256_kernel": page size a
 * constant 256, one page lookup per key tile).  max_rows_per_launch > 0 runs
 * the rows in slices of that many (a slice's result is the same bytes as one
 * launch); 0 = one launch.  bf16 and fp8 caches. */
int tfpa_prefill(const tfpa_cache* cache, const tfpa_seg* segs, int32_t nseg,
                 const void* q, const int32_t* row_seg, const int32_t* row_pos,
                 int32_t rows, float softmax_scale, int32_t max_rows_per_launch,
                 void* out, float* lse, cudaStream_t stream);

/* Launch recording for host tests (PR #1355: "a launch-recording host test
 * where a 257-row chunk issues 3 slices").  With a hook installed every
 * launch is reported; with dry_run != 0 nothing is enqueued and no CUDA call
 * is made, so the slicing logic runs on a machine without a GPU. */
typedef struct {
  int32_t kind;          /* 0 write_kv, 1 decode partial, 2 merge, 3 prefill, 4 keep,
                            5 stage pages, 6 save, 7 restore, 8 verify (decode or tree
                            rows of runs with 49 or more query vectors per kv head, on
                            tensor cores; items = tiles) */
  int32_t row0;          /* first row of the call this launch covers */
  int32_t rows;          /* rows it covers */
  int32_t runs;          /* row groups (segment, consecutive positions) */
  int32_t items;         /* work items (decode: tiles of (kv head, m-tile, split)) */
  int32_t grid;          /* CTAs (prefill: two per tile, in clusters of two) */
  int64_t q_offset;      /* element offset of the q pointer it got, from the call's q */
  int64_t out_offset;    /* element offset of the out pointer, from the call's out */
} tfpa_launch_record;
typedef void (*tfpa_launch_hook)(const tfpa_launch_record* rec, void* user);
void tfpa_set_launch_hook(tfpa_launch_hook hook, void* user, int dry_run);

const char* tfpa_strerror(int code);
const char* tfpa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TFPA_H */
