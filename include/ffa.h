/*
 * ffa.h -- C ABI of libffa.so: range-masked flash attention for GB300 (sm_103a).
 *
 * The operation is the one behind flex_flash_attn_func as described in MagiAttention issue
 * #180 ("Using dummy/padded attention slices with flex_flash_attn_func for torch.compile
 * static shapes", question code and maintainer reply): softmax attention over packed tokens
 * q:[Nq,Hq,d], k,v:[Nk,Hkv,d], masked by a list of slices (q_range, k_range, type), type
 * 0 = FULL and 1 = CAUSAL, returning out:[Nq,Hq,d] and the per-row log-sum-exp; the
 * backward pass returns dq, dk, dv.  A slice whose q-range or k-range has start == end
 * covers no area and is ignored (maintainer reply, "Mechanism").
 *
 * Semantics fixed by this library where the pages are silent:
 *   - CAUSAL is bottom-right aligned inside its slice: pair (i, j) of slice
 *     [qs,qe) x [ks,ke) is visible iff qs <= i < qe, ks <= j < ke and j <= i + ke - qe.
 *   - Overlapping slices combine by logical OR (union): a pair is counted once however many
 *     slices cover it (mask composition by logical operations, Flex Attention paper,
 *     section 3, "Composability").
 *   - softcap > 0: score x = softcap * tanh(softmax_scale * q.k / softcap); 0 disables it.
 *   - softmax_scale <= 0 or NaN selects 1/sqrt(d).
 *   - Rows with no visible key get out = 0 and lse = -inf; they contribute nothing to any
 *     gradient and their dq is 0.
 *   - lse is the natural-log log-sum-exp, float32, laid out [Hq, Nq].
 *   - GQA: query head h reads key/value head h / (Hq / Hkv).
 *
 * Conventions for every entry point:
 *   - Tensors are contiguous, row-major, bf16 unless stated; pointers marked "device" must
 *     be device (or managed) memory visible to the current device, 16-byte aligned.
 *   - The caller owns every buffer, including the workspace; the library keeps no device
 *     memory between calls.  All work is enqueued on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) without host synchronisation, so outputs are valid only after
 *     the stream has been synchronised.
 *   - Errors detectable on the host (null pointers, unsupported shapes, a workspace that is
 *     too small, misalignment) are returned before anything is launched.  Slice contents
 *     live on the device: a malformed slice (bound outside [0, N], start > end, unknown
 *     type) is dropped by the planner, which ORs FFA_STATUS_BAD_RANGE into *status.  A
 *     bounded wait inside a kernel that runs out ORs FFA_STATUS_TIMEOUT into *status.
 *     *status is a device int32 that the library only ORs into (the caller clears it);
 *     it may be NULL.
 *   - Environment, read on every call: FFA_WAIT_LIMIT_NS (decimal) bounds every wait inside
 *     a kernel (default 4 s).  FFA_TEST_STALL=1 is a failure-detection test switch: the first
 *     wait of every CTA of the forward and backward attention kernels then targets a barrier
 *     that nothing arrives on, so it runs out after FFA_WAIT_LIMIT_NS, the kernel records
 *     FFA_STATUS_TIMEOUT, lets its in-flight copies and MMAs land, frees its tensor memory and
 *     returns (outputs are then undefined).  Leave it unset in normal use.
 */
#ifndef FFA_H_
#define FFA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* return codes */
#define FFA_OK 0
#define FFA_ERR_INVALID_ARG 1 /* null pointer, bad shape, n_ranges < 0, misalignment   */
#define FFA_ERR_UNSUPPORTED 2 /* head_dim not in {64,128}, too many tokens, no sm_103a */
#define FFA_ERR_CUDA 3        /* a CUDA runtime/driver call failed                     */
#define FFA_ERR_WORKSPACE 4   /* workspace NULL or smaller than the *_workspace_size() */
#define FFA_ERR_TOO_LARGE 5   /* problem needs more scratch than ffa_fwd_noalloc owns  */

/* bits of the device status word */
#define FFA_STATUS_BAD_RANGE 1 /* a malformed slice was dropped                       */
#define FFA_STATUS_TIMEOUT 2   /* a bounded wait inside a kernel ran out              */
#define FFA_STATUS_SMEM 4      /* shared memory could not be aligned for the tiles    */
#define FFA_STATUS_BAD_PAGE 8  /* a page-table entry pointed outside the page pool    */

/* slice types (attn_type_map values) */
#define FFA_FULL 0
#define FFA_CAUSAL 1

/* tile classes written by ffa_plan_tiles */
#define FFA_TILE_EMPTY 0
#define FFA_TILE_PARTIAL 1
#define FFA_TILE_FULL 2
#define FFA_TILE_SIZE 128

/* largest supported total_q / total_k */
#define FFA_MAX_TOKENS (1 << 20)

typedef struct ffa_shape {
  int64_t total_q;      /* Nq: packed query tokens, 0 <= Nq <= FFA_MAX_TOKENS           */
  int64_t total_k;      /* Nk: packed key/value tokens, 0 <= Nk <= FFA_MAX_TOKENS       */
  int32_t num_heads_q;  /* Hq >= 1                                                      */
  int32_t num_heads_kv; /* Hkv >= 1, Hq % Hkv == 0                                      */
  int32_t head_dim;     /* d in {64, 128}                                               */
} ffa_shape;

/*
 * Bytes of workspace ffa_fwd / ffa_bwd / ffa_plan_tiles need for this shape and slice count.
 * The forward workspace holds the planner's output (compacted slices, the tile-class grid,
 * per-tile-row work lists and their longest-first order); it grows with
 * ceil(Nq/128) * ceil(Nk/128).  The backward workspace holds the column-wise plan plus the
 * float32 row statistic D [Hq, Nq] and the float32 dq accumulator [Nq, Hq, d].
 * Returns 0 for an invalid shape.
 */
size_t ffa_fwd_workspace_size(const ffa_shape* shape, int32_t n_ranges);
size_t ffa_bwd_workspace_size(const ffa_shape* shape, int32_t n_ranges);

/*
 * Forward pass: out, lse = attention(q, k, v, slices).  This is flex_flash_attn_func(q, k, v,
 * max_seqlen_q, max_seqlen_k, q_ranges, k_ranges, attn_type_map, softmax_scale, softcap) ->
 * (out, lse) of MagiAttention issue #180 (the reproduction script's attention call); the
 * max_seqlen arguments are not needed because tiles lie on the global grid of the packed
 * tensors.
 *   q        device bf16 [Nq, Hq, d]
 *   k, v     device bf16 [Nk, Hkv, d]
 *   q_ranges, k_ranges  device int32 [n_ranges, 2] (start, end) pairs, end exclusive
 *   attn_type_map       device int32 [n_ranges], FFA_FULL or FFA_CAUSAL
 *   n_ranges            >= 0 (0 means nothing is visible)
 *   softmax_scale       <= 0 or NaN -> 1/sqrt(d)
 *   softcap             0 disables; must be >= 0
 *   out      device bf16 [Nq, Hq, d], written
 *   lse      device float32 [Hq, Nq], written
 *   workspace, workspace_bytes  device scratch of at least ffa_fwd_workspace_size() bytes,
 *            256-byte aligned; contents on entry are ignored
 *   status   device int32 or NULL (see above)
 *   stream   cudaStream_t
 * Results are bit-identical from run to run and under appended start == end slices.
 */
int ffa_fwd(const ffa_shape* shape, const void* q, const void* k, const void* v, const int32_t* q_ranges,
            const int32_t* k_ranges, const int32_t* attn_type_map, int32_t n_ranges, float softmax_scale,
            float softcap, void* out, float* lse, void* workspace, size_t workspace_bytes, int32_t* status,
            void* stream);

/*
 * Backward pass: gradients of sum(out * dout) with respect to q, k and v, the dq/dk/dv that
 * MagiAttention issue #180's reproduction script obtains with out.backward(do).
 *   q, k, v, q_ranges, k_ranges, attn_type_map, n_ranges, softmax_scale, softcap: as for
 *            ffa_fwd (same values as the forward call)
 *   out      device bf16 [Nq, Hq, d]: the forward output
 *   lse      device float32 [Hq, Nq]: the forward log-sum-exp
 *   dout     device bf16 [Nq, Hq, d]
 *   dq       device bf16 [Nq, Hq, d], written
 *   dk, dv   device bf16 [Nk, Hkv, d], written
 *   workspace  at least ffa_bwd_workspace_size() bytes
 * dq is accumulated in a float32 buffer by TMA bulk reduce-adds from many CTAs, so its
 * summation order (and its last bits) may differ from run to run; dk and dv are written once
 * per (key tile, kv head).  ffa_bwd_ex with deterministic = 1 fixes the order.
 */
int ffa_bwd(const ffa_shape* shape, const void* q, const void* k, const void* v, const void* out,
            const float* lse, const void* dout, const int32_t* q_ranges, const int32_t* k_ranges,
            const int32_t* attn_type_map, int32_t n_ranges, float softmax_scale, float softcap, void* dq,
            void* dk, void* dv, void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/*
 * Optional score modification and future options for ffa_fwd_ex / ffa_bwd_ex.  A
 * zero-initialised struct (or a NULL pointer) means: none.
 *   alibi_slopes  device float32 [Hq] or NULL.  Adds slope_h * (j - i) to the (softcapped)
 *                 score of query position i and key position j (packed token indices; for
 *                 two tokens of one document this is their in-document distance): the ALiBi
 *                 distance bias, a score modification of the Flex Attention paper
 *                 (sections 2 and 3.1).  The bias enters the softmax only; it has no
 *                 gradient.  Pass the same slopes to the forward and backward calls.
 *   deterministic backward only.  Nonzero: each query tile's dq receives the contributions of
 *                 its key tiles in ascending key-tile order (a per-(head, query tile)
 *                 counter orders the float32 additions), so dq, dk and dv are bit-identical
 *                 from run to run and under appended start == end slices.  The backward
 *                 kernel then runs as a cooperative launch over key tiles in ascending
 *                 order; waits on the counters are bounded (FFA_STATUS_TIMEOUT).
 *   reserved      must be zero.
 */
typedef struct ffa_options {
  const float* alibi_slopes;
  int32_t deterministic;
  int32_t reserved[7];
} ffa_options;

/* ffa_fwd with options (NULL options: identical to ffa_fwd). */
int ffa_fwd_ex(const ffa_shape* shape, const void* q, const void* k, const void* v, const int32_t* q_ranges,
               const int32_t* k_ranges, const int32_t* attn_type_map, int32_t n_ranges, float softmax_scale,
               float softcap, void* out, float* lse, void* workspace, size_t workspace_bytes, int32_t* status,
               void* stream, const ffa_options* options);

/* ffa_bwd with options (NULL options: identical to ffa_bwd). */
int ffa_bwd_ex(const ffa_shape* shape, const void* q, const void* k, const void* v, const void* out,
               const float* lse, const void* dout, const int32_t* q_ranges, const int32_t* k_ranges,
               const int32_t* attn_type_map, int32_t n_ranges, float softmax_scale, float softcap, void* dq,
               void* dk, void* dv, void* workspace, size_t workspace_bytes, int32_t* status, void* stream,
               const ffa_options* options);

/*
 * Forward pass over a paged key/value cache (FlexAttention paper, section 5, Paged
 * Attention: a shared physical cache indexed through a page table, with masks written in
 * logical positions).  Slices, masks, ALiBi and all results use logical key positions
 * 0 .. shape->total_k - 1 exactly as ffa_fwd does; only where a key's data lives differs.
 *   k_pages, v_pages  device bf16 [n_pages, page_size, Hkv, d], 16-byte aligned: the pool
 *   page_table        device int32 [ceil(total_k / page_size)]: logical page j of the key
 *                     sequence (keys j*page_size .. j*page_size + page_size - 1) is
 *                     physical page page_table[j].  Pages may be shared or unused.
 *   page_size         16, 32, 64 or 128 keys
 *   n_pages           pages in the pool, >= 1, n_pages * page_size < 2^31
 *   options           as for ffa_fwd_ex (deterministic has no effect on a forward pass)
 * Other arguments, the workspace size and the results are those of ffa_fwd (same
 * ffa_fwd_workspace_size()).  An entry outside [0, n_pages) makes its keys read as zeros
 * and ORs FFA_STATUS_BAD_PAGE into *status.  Forward only: gradients through a paged cache
 * are not provided.
 */
int ffa_fwd_paged(const ffa_shape* shape, const void* q, const void* k_pages, const void* v_pages,
                  const int32_t* page_table, int32_t page_size, int64_t n_pages, const int32_t* q_ranges,
                  const int32_t* k_ranges, const int32_t* attn_type_map, int32_t n_ranges, float softmax_scale,
                  float softcap, void* out, float* lse, void* workspace, size_t workspace_bytes, int32_t* status,
                  void* stream, const ffa_options* options);

/*
 * Decoding: few new query tokens per sequence against long (optionally paged) key caches
 * (FlexAttention paper: a decoding template with grouped-query attention support, section
 * 4; decoding measured against FlashDecoding, section 6).  Same arguments and results as
 * ffa_fwd (page_table == NULL) or ffa_fwd_paged (page_table != NULL), plus
 *   max_seqlen_q  >= 1: the most query tokens any CAUSAL slice has (the max_seqlen_q
 *                 argument of flex_flash_attn_func); a CAUSAL slice with more is dropped and
 *                 reported with FFA_STATUS_BAD_RANGE
 * The G = Hq / Hkv query heads of every token are processed as G rows of the key/value head
 * they share, so each key tile is read once per (128-row query tile, key/value head) and
 * multiplied once, by alternating halves of the work item (the forward pass's key split).
 * options->alibi_slopes
 * ([Hq], as for ffa_fwd_ex) gives every query head its own slope and every token its own
 * position, exactly as in the unpacked problem.  Requires total_q * G <= FFA_MAX_TOKENS.
 * workspace: ffa_fwd_decode_workspace_size() bytes.
 */
size_t ffa_fwd_decode_workspace_size(const ffa_shape* shape, int32_t n_ranges, int32_t max_seqlen_q);
int ffa_fwd_decode(const ffa_shape* shape, const void* q, const void* k, const void* v, const int32_t* page_table,
                   int32_t page_size, int64_t n_pages, const int32_t* q_ranges, const int32_t* k_ranges,
                   const int32_t* attn_type_map, int32_t n_ranges, int32_t max_seqlen_q, float softmax_scale,
                   float softcap, void* out, float* lse, void* workspace, size_t workspace_bytes, int32_t* status,
                   void* stream, const ffa_options* options);

/*
 * The planner alone: classify every tile of the global 128 x 128 tile grid as
 * FFA_TILE_EMPTY / PARTIAL / FULL under the union of the slices (block classification of
 * the Flex Attention paper, section 4, "Block Sparsity" / "Full Block Optimization"),
 * restricted to in-bounds entries.
 *   tile_class  device uint8 [ceil(Nq/128), ceil(Nk/128)], written
 *   by_column   0: the forward planner (one pass per query-tile row);
 *               1: the backward planner (one pass per key-tile column)
 *   workspace   at least ffa_fwd_workspace_size() (by_column = 0) or
 *               ffa_bwd_workspace_size() (by_column = 1) bytes
 */
int ffa_plan_tiles(const ffa_shape* shape, const int32_t* q_ranges, const int32_t* k_ranges,
                   const int32_t* attn_type_map, int32_t n_ranges, int32_t by_column, uint8_t* tile_class,
                   void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/*
 * Measurement hook.  When the handles are non-NULL, each later ffa_fwd call records
 * fwd_start on its stream immediately before the forward attention kernel and fwd_stop
 * immediately after it (the planner launches stay outside the pair); ffa_bwd does the same
 * around its main backward kernel with bwd_start / bwd_stop.  The handles are cudaEvent_t
 * created and owned by the caller; pass NULLs to stop recording.  The setting is
 * process-wide and not synchronised between threads.  Returns FFA_OK.
 */
int ffa_set_kernel_events(void* fwd_start, void* fwd_stop, void* bwd_start, void* bwd_stop);

/*
 * Forward pass for callers that cannot allocate device memory at call time (for example a
 * runtime that reserves all device memory up front and forbids later cudaMalloc, or a
 * latency-bound path that cannot afford the device synchronisation an allocation may
 * cause).  The pages describe no such variant: this entry point has no counterpart there.
 *
 * Same arguments and results as ffa_fwd, without the workspace.  The planner's scratch
 * lives in a fixed device array of FFA_FWD_NOALLOC_SCRATCH_BYTES owned by the library; it
 * exists once on every device that loads the library and stays allocated until the process
 * exits.  The function itself allocates nothing (no cudaMalloc, cudaFree or allocating
 * library routine).  The first call on a device looks up the array's device address with
 * that device current; make that first call before any stream capture.
 *   Returns FFA_ERR_TOO_LARGE (before launching anything) when ffa_fwd_workspace_size()
 *   for the shape exceeds FFA_FWD_NOALLOC_SCRATCH_BYTES, e.g. beyond about 160K tokens
 *   with a single query and key range.
 * Every call uses the same array and the planner overwrites everything it reads, so
 * nothing has to start at zero; calls whose kernels overlap on the GPU (other streams or
 * other host threads on the same device) race on the array and must be serialised.
 */
#define FFA_FWD_NOALLOC_SCRATCH_BYTES (8u << 20)
int ffa_fwd_noalloc(const ffa_shape* shape, const void* q, const void* k, const void* v,
                    const int32_t* q_ranges, const int32_t* k_ranges, const int32_t* attn_type_map,
                    int32_t n_ranges, float softmax_scale, float softcap, void* out, float* lse,
                    int32_t* status, void* stream);

/* Static description of a return code; never NULL. */
const char* ffa_status_string(int code);

/* Build description: target architecture, tile sizes, pipeline depths. */
const char* ffa_build_info(void);

#ifdef __cplusplus
}
#endif

#endif /* FFA_H_ */
