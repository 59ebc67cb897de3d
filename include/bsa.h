/*
 * bsa.h -- C ABI of a GB300 (sm_103a) block-sparse ("splash") attention library.
 *
 * The method: "Splash Attention: When the Mask Stops Being Arithmetic and
 * Becomes the Loop" (explainers.rudrite.com/splash-attention).  A mask is
 * compiled once into MaskInfo -- one label per block (0 = all zeros, never
 * computed or fetched; 1 = mixed, computed and masked; 2 = all ones,
 * computed without masking), the next non-empty key/value block per grid
 * position (data_next), a deduplicated stack of the mixed blocks of a dense
 * mask (partial_mask_blocks, pointed at by mask_next), the query indices
 * (q_sequence) -- and the attention kernels take their loop structure from
 * it.  The backward pass follows "Flash Attention on a TPU, Line by Line"
 * (explainers.rudrite.com/pallas-flash-attention-tpu): rowsum(dO*O) is
 * computed once by its own kernel, then one launch produces dK/dV (queries
 * innermost) and another dQ (keys innermost), both rebuilding the scores
 * from Q, K and the saved per-row logsumexp.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Tensors are contiguous BHSD: Q, O, dO, dQ are [B, Hq, S_q, D];
 *   K, V, dK, dV are [B, Hkv, S_kv, D]; LSE and Dsum are [B, Hq, S_q] fp32.
 *   Q/K/V/O/dO are bf16.  Query head h reads key/value head
 *   h / (Hq / Hkv) (contiguous groups: MHA, GQA and MQA).
 * - All tensor pointers are DEVICE pointers owned by the caller, 16-byte
 *   aligned.  The library never frees them.
 * - Blocks are 128 x 128; S_q and S_kv must be multiples of 128; D is 64 or
 *   128.
 * - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *   is asynchronous on that stream except bsa_mask_compile (which
 *   synchronises `stream` to learn the grid width and the stack size, and
 *   before it returns), bsa_mask_info_destroy and bsa_get_device_error.
 * - Calls return a status; none throws.  On failure bsa_last_error()
 *   returns a message for the calling thread.  Argument errors are found on
 *   the host before anything is launched.
 * - Kernels never trap: every device-side wait is bounded; a wait that runs
 *   out, or an index read from MaskInfo that is out of range, sets a bit in
 *   the library's device error word and the kernel returns.  Read it with
 *   bsa_get_device_error.
 */
#ifndef BSA_H_
#define BSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define BSA_API __attribute__((visibility("default")))
#else
#define BSA_API
#endif

typedef void* bsa_stream; /* a cudaStream_t */

typedef enum {
  BSA_OK = 0,
  BSA_ERR_INVALID_ARG = 1, /* null pointer, bad shape, S % 128 != 0, Hq % Hkv != 0, wrong MaskInfo */
  BSA_ERR_UNSUPPORTED = 2, /* D not in {64, 128}, block != 128, S_q != S_kv for a computable mask */
  BSA_ERR_CUDA = 3,        /* a CUDA runtime call failed (message in bsa_last_error) */
  BSA_ERR_OOM = 4,         /* the library could not allocate MaskInfo storage */
  BSA_ERR_TIMEOUT = 5,     /* a kernel's bounded wait ran out (device error word) */
  BSA_ERR_DEVICE = 6       /* a kernel found an out-of-range MaskInfo index (device error word) */
} bsa_status;

/* Mask kinds ("What is MaskInfo in splash attention?": CausalMask, LocalMask,
 * ChunkedCausalMask are computable; a dense array is materialised). */
typedef enum {
  BSA_MASK_DENSE = 0,          /* dense uint8 0/1 array (nonzero = visible)          */
  BSA_MASK_CAUSAL = 1,         /* k <= q                                             */
  BSA_MASK_LOCAL = 2,          /* q - left <= k <= q + right (inclusive; -1 = none)  */
  BSA_MASK_CHUNKED_CAUSAL = 3, /* q / chunk == k / chunk  and  k <= q               */
  BSA_MASK_FULL = 4            /* every key visible                                  */
} bsa_mask_kind;

typedef enum {
  BSA_ORIENT_FWD = 0, /* rows = query blocks, columns = key blocks (forward and dQ grids) */
  BSA_ORIENT_DKV = 1  /* rows = key blocks, columns = query blocks (dK/dV grid)           */
} bsa_orientation;

typedef struct {
  int32_t kind;          /* bsa_mask_kind */
  int32_t mask_heads;    /* 1 (shared by every query head) or Hq (one mask per query head) */
  int64_t q_len, kv_len; /* element sizes of the mask */
  int64_t local_left;    /* LOCAL: keys back to q - local_left are visible; -1 = unbounded */
  int64_t local_right;   /* LOCAL: keys up to q + local_right are visible; -1 = unbounded */
  int64_t chunk;         /* CHUNKED_CAUSAL: chunk length in tokens (> 0) */
  const uint8_t* dense;  /* DENSE: device [mask_heads, q_len, kv_len] uint8, caller-owned;
                            only read during bsa_mask_compile */
} bsa_mask_spec;

typedef struct {
  int32_t block_q;     /* must be 128 */
  int32_t block_kv;    /* must be 128 */
  int32_t shrink;      /* 1: apply the grid-shrink pass; 0: keep the full grid width */
  int32_t orientation; /* bsa_orientation */
} bsa_mask_opts;

/* Opaque compiled mask; owned by the library, freed by bsa_mask_info_destroy. */
typedef struct bsa_mask_info bsa_mask_info;

/* A read-only view of a compiled MaskInfo.  Device pointers stay valid until
 * bsa_mask_info_destroy.  Integer element sizes are 1, 2 or 4 bytes: each
 * array takes the smallest signed type its largest value fits in. */
typedef struct {
  const int8_t* block_mask;           /* [heads, rows, width] labels 0/1/2 */
  const void* data_next;              /* [heads, rows, width] key-block (fwd) / query-block (dkv) index */
  int32_t data_next_bytes;            /* 1, 2 or 4 */
  const void* mask_next;              /* [heads, rows, width] stack slot; NULL for computable masks */
  int32_t mask_next_bytes;            /* 1, 2 or 4 (0 if mask_next is NULL) */
  const uint8_t* partial_mask_blocks; /* [num_partial, 128, 128] 0/1; NULL for computable masks */
  const int32_t* q_sequence;          /* [q_len] the query indices */
  int32_t heads, rows, width, cols;   /* width = grid width after shrink; cols = before */
  int64_t num_partial;                /* P, the stack depth */
  int64_t n_empty, n_partial, n_full; /* block counts over the unshrunk grid, all heads */
  int32_t kind, orientation, shrink;
  int64_t q_len, kv_len;
  /* the library's own row arrays (beside MaskInfo proper, from which the
   * launches build their tile schedules): non-empty blocks per mask row,
   * and the rows by decreasing length, ties in increasing row order */
  const int32_t* row_len;             /* [heads * rows] */
  const int32_t* row_order;           /* [heads * rows] */
} bsa_mask_info_desc;

/* Compile a mask into MaskInfo ("What is MaskInfo in splash attention?",
 * "What does grid shrinking do in splash attention?").  Runs the classifier,
 * the partial-block dedup (dense masks only), the next-block pass, the
 * shrink pass and the integer downcast as kernels on `stream`, synchronising
 * `stream` to size the outputs and again before returning: the MaskInfo is
 * complete on return, and the attention kernels read it without waiting for
 * earlier work on their stream.  Its device memory (and the compile's
 * scratch) comes from a stream-ordered memory pool the library keeps per
 * device, so no step of the compile synchronises the whole device.  The
 * counts and row arrays the host needs come back through a pinned, mapped
 * host buffer that a kernel writes (no copy-engine transfer), so the compile
 * does not wait behind large host<->device copies other streams have in
 * flight.  *out receives a new handle on success and is untouched on
 * failure. */
BSA_API bsa_status bsa_mask_compile(const bsa_mask_spec* spec, const bsa_mask_opts* opts, bsa_stream stream,
                            bsa_mask_info** out);
BSA_API bsa_status bsa_mask_info_view(const bsa_mask_info* info, bsa_mask_info_desc* out);
/* Returns the handle's device storage to the library's pool (synchronises
 * the device first, so no launch still reads it). NULL is accepted. */
BSA_API bsa_status bsa_mask_info_destroy(bsa_mask_info* info);

typedef struct {
  const void* q;       /* bf16 [B, Hq, S_q, D] */
  const void* k;       /* bf16 [B, Hkv, S_kv, D] */
  const void* v;       /* bf16 [B, Hkv, S_kv, D] */
  void* o;             /* bf16 [B, Hq, S_q, D], written */
  float* lse;          /* fp32 [B, Hq, S_q], written: natural-log logsumexp of the scaled
                          scores of each row (-inf for a row with no visible key) */
  int32_t B, Hq, Hkv, D;
  int64_t S_q, S_kv;
  float softmax_scale; /* NaN selects 1/sqrt(D) */
  /* Optional score transforms (the logits_soft_cap and softmax_aux arguments
   * of the EasyDeL blocksparse_attention operator; zero-initialised = off):
   * logits_soft_cap c > 0 maps each visible scaled score s to c*tanh(s/c);
   * sinks are num_sinks extra logits per row that enter the normaliser (and
   * the maximum) but carry no value, fp32 on the device, [Hkv, num_sinks]
   * (q head h uses row h / (Hq/Hkv)) when sinks_per_kv_head is 1, else
   * [num_sinks] shared by all heads.  LSE includes the sinks; a row with no
   * visible key gets O = 0 and LSE = log(sum_j exp(z_j)). */
  float logits_soft_cap;
  const float* sinks;
  int32_t num_sinks;   /* 0..64 */
  int32_t sinks_per_kv_head;
} bsa_fwd_args;

/* Block-sparse forward ("What is splash attention and how is it different
 * from flash attention?"): for every (b, query head, query block) the kernel
 * walks the MaskInfo row, never fetches or computes label-0 blocks, masks
 * only label-1 blocks, and runs an online softmax (running max and sum, one
 * divide at the end).  `fwd_info` must be a BSA_ORIENT_FWD MaskInfo with
 * q_len == S_q, kv_len == S_kv and mask_heads 1 or Hq.  A query row with no
 * visible key gets O = 0 and LSE = -inf.  The kernel is launched with
 * programmatic stream serialization: its set-up overlaps the end of the
 * previous kernel on `stream`, and it waits for that kernel before reading
 * Q/K/V or writing O/LSE (BSA_PDL=0 in the environment turns this off).
 * The first launch of a (B, Hq, SM count) configuration builds its tile
 * schedule on the host (kept for the process per row lengths and
 * configuration, so a mask compiled again reuses it) and uploads it in
 * stream order on `stream`, in the parameters of small copy kernels rather
 * than through a copy engine, so that it never waits behind other streams'
 * host<->device copies (cached in the MaskInfo; a later launch on another
 * stream waits for the upload through an event). */
BSA_API bsa_status bsa_fwd(const bsa_fwd_args* args, const bsa_mask_info* fwd_info, bsa_stream stream);

/* One shard of the key axis ("Splash Attention: When the Mask Stops Being
 * Arithmetic and Becomes the Loop", "What does ring attention add on top of
 * the splash kernel?"): the keys and values are split into shards, each
 * shard's attention runs with the MaskInfo cut to the shard's key range,
 * and the per-shard results are merged with the flash rescaling
 * (bsa_fwd_merge).  The shard's K and V are given on their own; the
 * MaskInfo is the one for the whole key axis. */
typedef struct {
  const void* q;        /* bf16 [B, Hq, S_q, D] */
  const void* k;        /* bf16 [B, Hkv, S_kv_shard, D]: keys kv_offset .. kv_offset + S_kv_shard - 1 */
  const void* v;        /* bf16 [B, Hkv, S_kv_shard, D] */
  float* o_acc;         /* fp32 [B, Hq, S_q, D], written: sum over the shard's visible keys of
                           exp(s - m) v (0 for a row with no visible key in the shard) */
  float* m;             /* fp32 [B, Hq, S_q], written: the row's reference maximum of the scaled
                           scores, natural-log units (-inf for a row with no visible key); it may
                           lag the true maximum by up to 8 log2 units: only m + log(l) and
                           o_acc / l are determined */
  float* l;             /* fp32 [B, Hq, S_q], written: sum over the shard's visible keys of exp(s - m) */
  int32_t B, Hq, Hkv, D;
  int64_t S_q;
  int64_t S_kv_shard;   /* multiple of 128 */
  int64_t kv_offset;    /* the shard's first key on the MaskInfo's key axis, multiple of 128 */
  float softmax_scale;  /* NaN selects 1/sqrt(D) */
  float logits_soft_cap; /* as in bsa_fwd_args (sinks are not accepted for shards: they would
                            enter every shard's normaliser) */
} bsa_fwd_partial_args;

/* Forward over one key shard: the same kernel as bsa_fwd, walking only the
 * MaskInfo blocks whose key block lies in [kv_offset, kv_offset + S_kv_shard)
 * and writing the unnormalised accumulator, maximum and normaliser instead
 * of O and LSE.  Requires kv_offset + S_kv_shard <= the MaskInfo's kv_len. */
BSA_API bsa_status bsa_fwd_partial(const bsa_fwd_partial_args* args, const bsa_mask_info* fwd_info,
                                   bsa_stream stream);

typedef struct {
  int32_t n_shards;     /* >= 1 */
  const float* o_acc;   /* fp32 [n_shards, rows, D]: the shards' o_acc, one after the other */
  const float* m;       /* fp32 [n_shards, rows] */
  const float* l;       /* fp32 [n_shards, rows] */
  void* o;              /* bf16 [rows, D], written: sum_i exp(m_i - M) o_acc_i / L */
  float* lse;           /* fp32 [rows], written: M + log L (-inf when every shard is empty) */
  int64_t rows;         /* B * Hq * S_q */
  int32_t D;
} bsa_merge_args;

/* Merge of key shards (same section): M = max of the shards' m over shards
 * with l > 0, L = sum_i exp(m_i - M) l_i, one final divide.  A shard that is
 * empty for a row (l = 0) contributes nothing; a row empty in every shard
 * gets O = 0 and LSE = -inf. */
BSA_API bsa_status bsa_fwd_merge(const bsa_merge_args* args, bsa_stream stream);

typedef struct {
  const void* q, *k, *v; /* as in bsa_fwd_args */
  const void* o;         /* bf16 forward output */
  const float* lse;      /* fp32 forward logsumexp */
  const void* do_;       /* bf16 [B, Hq, S_q, D] incoming gradient */
  void* dq;              /* [B, Hq, S_q, D], written; bf16 or fp32 per grad_fp32 */
  void* dk;              /* [B, Hkv, S_kv, D], written (summed over each query-head group) */
  void* dv;              /* [B, Hkv, S_kv, D], written (summed over each query-head group) */
  float* dsum;           /* caller-provided workspace fp32 [B, Hq, S_q]: rowsum(dO*O) */
  int32_t B, Hq, Hkv, D;
  int64_t S_q, S_kv;
  float softmax_scale;   /* NaN selects 1/sqrt(D) */
  int32_t grad_fp32;     /* 0: dq/dk/dv are bf16; 1: fp32 */
  /* The forward's score transforms (see bsa_fwd_args); lse must come from a
   * forward with the same ones.  With the cap, dS is taken through
   * c*tanh(s/c) (times 1 - tanh^2).  With sinks and a non-null dsinks, the
   * sinks' gradient -sum over rows of exp(z_j - LSE) * Dsum is written to
   * dsinks (fp32, the sinks' shape; accumulated with atomics, so the
   * summation order, and the last bits, vary between runs). */
  float logits_soft_cap;
  const float* sinks;
  float* dsinks;
  int32_t num_sinks;
  int32_t sinks_per_kv_head;
} bsa_bwd_args;

/* Backward ("Flash Attention on a TPU, Line by Line": "Why does the TPU flash
 * attention backward pass run two kernels instead of one?", "What does the
 * TPU flash attention kernel save for the backward pass?").  Runs
 * bsa_bwd_rowsum, then bsa_bwd_dkv with `dkv_info` (a BSA_ORIENT_DKV
 * MaskInfo of the same mask), then bsa_bwd_dq with `fwd_info`. */
BSA_API bsa_status bsa_bwd(const bsa_bwd_args* args, const bsa_mask_info* fwd_info, const bsa_mask_info* dkv_info,
                   bsa_stream stream);
/* dsum[b,h,s] = sum_d dO[b,h,s,d] * O[b,h,s,d] (fp32); with sinks and
 * dsinks, also the sinks' gradient (it needs Dsum and LSE only). */
BSA_API bsa_status bsa_bwd_rowsum(const bsa_bwd_args* args, bsa_stream stream);
/* dK, dV: grid over (b, kv head, key block), queries innermost.  When
 * B * Hkv * (S_kv / 128) is small next to the number of SMs (MQA, short
 * sequences) the q heads of each group are split over several CTAs: their
 * fp32 partial sums go to stream-ordered workspace taken from a memory pool
 * the library keeps per device (cudaMallocFromPoolAsync, returned with
 * cudaFreeAsync on `stream`, kept cached by the pool) and a second kernel
 * adds them up in a fixed order.  The first launch of a configuration also
 * builds its tile schedule (uploaded in stream order, cached in the
 * MaskInfo, as for bsa_fwd); bsa_bwd_noalloc does neither. */
BSA_API bsa_status bsa_bwd_dkv(const bsa_bwd_args* args, const bsa_mask_info* dkv_info, bsa_stream stream);
/* dQ: grid over (b, query head, query block), keys innermost.  The first
 * launch of a configuration builds its tile schedule (cached in the MaskInfo,
 * shared with bsa_fwd). */
BSA_API bsa_status bsa_bwd_dq(const bsa_bwd_args* args, const bsa_mask_info* fwd_info, bsa_stream stream);

/* The backward pass (rowsum, dK/dV, dQ, same arguments and results as
 * bsa_bwd) without allocating any device memory, for callers that cannot
 * allocate: a runtime whose device memory is fixed up front by its own pool
 * or budget, or a latency-critical loop that must not hit the device-wide
 * synchronisation an allocation or free can cause.  The splash-attention
 * pages have no counterpart; it is an addition of this library.
 *   - args->dsum is ignored: the rowsum(dO*O) scratch is a file-scope device
 *     array of 1,048,576 fp32 (4 MiB) that every GPU loading the library
 *     holds until the process exits.  B * Hq * S_q above 1,048,576 is
 *     rejected with BSA_ERR_UNSUPPORTED before anything is launched.
 *   - The first call on a device looks up the array's device address for
 *     that device (cudaGetSymbolAddress, with that device current); make
 *     that first call before any stream capture.
 *   - Every call shares the one array (and keeps the last call's rowsum in
 *     it): calls that overlap on the GPU race, so serialise them (one
 *     stream, or events).
 *   - Device-side error bits of this entry point (a wait that ran out, a bad
 *     MaskInfo index) go to a device word of its own, also static; they
 *     stay set until bsa_get_device_error reads and clears them (it reads
 *     this word together with the library's own and allocates neither).
 *     Host-side argument errors are returned as for bsa_bwd, with the same
 *     checks (pointer alignment, sinks and dsinks included) except that
 *     args->dsum is not looked at. */
BSA_API bsa_status bsa_bwd_noalloc(const bsa_bwd_args* args, const bsa_mask_info* fwd_info,
                                   const bsa_mask_info* dkv_info, bsa_stream stream);

/* Synchronises `stream`, returns the device error word of the current
 * device in *word and clears it.  0 = none; otherwise an OR of the flags
 * 1 = a bounded wait ran out, 2 = out-of-range MaskInfo index, 4 =
 * tensor-memory allocation failure, 8 = a check of the range-checked build
 * (the source line of the first one is then in bits 16-31 of the word),
 * 16 = a kernel found its dynamic shared memory off the 1024-byte boundary
 * it is laid out for, and did nothing.  The word is the OR of the
 * library's word (set by every launch but those of bsa_bwd_noalloc) and
 * bsa_bwd_noalloc's own; a word no launch has set up yet reads as 0, and
 * nothing is allocated here.  The status is BSA_ERR_TIMEOUT /
 * BSA_ERR_DEVICE when the word is non-zero. */
BSA_API bsa_status bsa_get_device_error(bsa_stream stream, uint32_t* word);

/* Time limit of one device-side wait, in nanoseconds (default 2e9).  Applies
 * to launches made after the call.  0 restores the default. */
BSA_API bsa_status bsa_set_wait_limit_ns(uint64_t ns);

/* Launches one CTA that waits on an mbarrier nothing ever arrives at, with
 * the current wait limit, and returns.  Used to check that a wait that runs
 * out ends with BSA_ERR_TIMEOUT in the device error word instead of a hang. */
BSA_API bsa_status bsa_debug_wait_timeout(bsa_stream stream);

/* Launches one thread that passes out-of-range indices through the kernels'
 * range checks.  In the range-checked build of the library (libbsa_debug.so,
 * compiled with -DBSA_DEBUG=1: tensor-memory addresses, the global rows the
 * kernels compute and the phases of mbarriers are checked on the device)
 * the device error word then holds bit 8 (DEV_ERR_DEBUG) with the source
 * line of the first violation in bits 16-31; in the release build the
 * checks are compiled out and the word stays 0.  Used to check that the
 * range-checked build reports what it finds. */
BSA_API bsa_status bsa_debug_selfcheck(bsa_stream stream);

/* The launch-time tile schedule of the persistent attention launches, as
 * they build it on the host (a testing aid: no device work, no GPU needed).
 * Inputs as a MaskInfo holds them: row_len[heads * rows] (non-empty blocks
 * per mask row) and row_order[rows] (rows by decreasing length; read only
 * when heads == 1).  Tiles are (batch of n_b, group g of n_g, mask row,
 * split) with `group` mask heads per group split in `splits` (the forward
 * and dQ launches: n_g = Hq, group = splits = 1; dK/dV: n_g = Hkv, group =
 * Hq / Hkv).  They are assigned longest first, each to the CTA of the
 * `grid` with the least work so far (ties to the lower index; a tile of n
 * blocks costs 8n + 12).  Writes CTA c's list at out[(c * cap + k) * 4 +
 * {0..3}] = {row, blocks, b * n_g + g, split}, closed by an entry with
 * blocks = -1 and padded with such entries, and *stride = the longest list
 * + 1; BSA_ERR_INVALID_ARG (with *stride set) when cap < *stride. */
BSA_API bsa_status bsa_debug_tile_schedule(const int32_t* row_len, const int32_t* row_order, int32_t rows,
                                           int32_t heads, int32_t n_b, int32_t n_g, int32_t group,
                                           int32_t splits, int32_t grid, int32_t* out, int32_t cap,
                                           int32_t* stride);

BSA_API const char* bsa_status_string(bsa_status s);
BSA_API const char* bsa_last_error(void);
/* Library version, e.g. "0.1.0". */
BSA_API const char* bsa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* BSA_H_ */
