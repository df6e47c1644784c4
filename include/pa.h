/*
 * pa.h -- C ABI of libpa: paged KV-cache append and single-query decode
 * attention for NVIDIA GB300 (sm_103a), plus the host block manager that
 * produces block tables and slot mappings.
 *
 * Sources (web pages on PagedAttention):
 *   [VM]  "PagedAttention: Virtual Memory Guide for LLM Inference"
 *   [MW]  "Solving the LLM Memory Wall: A Deep Dive into PagedAttention"
 *   [SE]  "PagedAttention, simply explained"
 *
 * Conventions shared by every call:
 *   - Return value: PA_OK (0) on success, a positive PA_WARN_* for a tolerated
 *     no-op, a negative PA_ERR_* on failure.  A failing call changes nothing
 *     (host state) and launches nothing (device).  pa_strerror() names a code.
 *   - Tensors are described by pa_tensor (data pointer, dtype, shape, strides in
 *     ELEMENTS).  The caller owns all tensor memory.  Device calls take device
 *     pointers; pa_bm_* calls take host pointers.
 *   - Device calls are asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).  They bounds-check indices read from device memory
 *     (slots, block ids, context lengths); a bad index is skipped (and for
 *     decode the affected output rows are written as zeros) and a bit is set in a
 *     sticky per-device status word that pa_get_device_status() reads.  No kernel
 *     traps or asserts.
 *   - Cache layout [MW "The Architecture at a Glance"]: k_cache and v_cache are
 *     separate contiguous tensors [num_blocks, block_size, num_heads, head_dim];
 *     token i of a sequence sits at frame table[i / block_size], offset
 *     i % block_size [VM "The Mathematics of Block Translation"]; its flat slot is
 *     frame * block_size + offset.  head_dim * element size must be a multiple of
 *     16 bytes and num_blocks * block_size must fit in int32.
 */
#ifndef PA_H_
#define PA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- element types ---------------------------------------------------------------- */
enum pa_dtype { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2, PA_I32 = 3 };

/* ---- return codes ------------------------------------------------------------------ */
#define PA_OK                 0
#define PA_WARN_DOUBLE_FREE   1   /* pa_bm_free of a sequence that is not live: no-op */
#define PA_ERR_INVALID       -1   /* null pointer, negative count, bad option */
#define PA_ERR_DTYPE         -2
#define PA_ERR_SHAPE         -3
#define PA_ERR_STRIDE        -4
#define PA_ERR_ALIGN         -5
#define PA_ERR_OUT_OF_BLOCKS -6   /* free list cannot cover the request (state unchanged) */
#define PA_ERR_UNKNOWN_SEQ   -7
#define PA_ERR_SEQ_EXISTS    -8
#define PA_ERR_CUDA          -9   /* a CUDA runtime call or launch failed */
#define PA_ERR_UNSUPPORTED  -10   /* head_dim / dtype / size outside the built kernels */
#define PA_ERR_CAPACITY     -11   /* caller-provided output buffer too small */
#define PA_ERR_SCRATCH_LIMIT -12  /* pa_decode_static: scratch need exceeds its fixed array */
#define PA_ERR_HOST_MEMORY  -13   /* a host allocation failed (no exception crosses this ABI) */

/* ---- sticky device status bits (pa_get_device_status) ------------------------------ */
#define PA_DEV_BAD_SLOT   0x1   /* append: slot >= num_blocks*block_size */
#define PA_DEV_BAD_BLOCK  0x2   /* decode: block-table entry outside [0, num_blocks) */
#define PA_DEV_BAD_LEN    0x4   /* decode: context_len < 0 or > max_blocks*block_size */
#define PA_DEV_BAD_COPY   0x8   /* copy_blocks: frame id outside [0, num_blocks) */
#define PA_DEV_TIMEOUT    0x10  /* a bounded wait inside a kernel gave up */

typedef struct pa_tensor {
  void*   data;       /* device (or host, where stated) pointer to element [0,...,0] */
  int32_t dtype;      /* enum pa_dtype */
  int32_t ndim;       /* 1..4 */
  int64_t shape[4];
  int64_t stride[4];  /* in elements */
} pa_tensor;

typedef void* pa_stream;   /* cudaStream_t */

/* ===================================================================================
 * Device path
 * =================================================================================== */

/*
 * pa_cache_append -- write each new token's K and V rows into its paged slot.
 * [MW "Implementation", PagedKVCache.update, batched over tokens; VM "Key
 * Architectural Mechanics / 1. Demand Paging": the token lands at offset t mod B
 * of its current frame, no reallocation or data movement.]
 *
 *   k_new, v_new   [T, H, D] (q/cache dtype); the [H, D] part contiguous, row
 *                  stride (stride[0]) free but a multiple of 16 bytes.
 *   slot_mapping   int32 [T]; k_cache.view(-1, H, D)[slot[t]] = k_new[t] (same for
 *                  v).  slot < 0 = padding, skipped.  slot >= num_blocks*B sets
 *                  PA_DEV_BAD_SLOT and is skipped.
 *   k_cache, v_cache  [num_blocks, B, H, D], contiguous, same dtype as k_new.
 * Slots within one call must be distinct (each is written by one thread block,
 * in no particular order).  T == 0 is a no-op.
 */
int pa_cache_append(const pa_tensor* k_new, const pa_tensor* v_new,
                    const pa_tensor* slot_mapping,
                    const pa_tensor* k_cache, const pa_tensor* v_cache,
                    pa_stream stream);

/*
 * pa_copy_blocks -- whole-frame copies for copy-on-write.
 * [VM "Key Architectural Mechanics / 2. Zero-Copy Branching via Copy-on-Write":
 * only the one shared frame being written is duplicated.]
 *
 *   pairs   int32 [n, 2], row = (src frame, dst frame); contiguous.  Both caches
 *           get cache[dst] = cache[src].  Ids outside [0, num_blocks) set
 *           PA_DEV_BAD_COPY and the pair is skipped.  Destinations must be
 *           distinct and no destination may be another pair's source.
 * Issue a decode step's copies BEFORE that step's pa_cache_append.
 */
int pa_copy_blocks(const pa_tensor* k_cache, const pa_tensor* v_cache,
                   const pa_tensor* pairs, pa_stream stream);

/*
 * pa_decode -- single-query decode attention over the paged cache.
 * [MW "1. The Mathematical Foundation": a_j = q.k_j * scale, o = sum_j softmax(a)_j
 *  v_j over the sequence's tokens; VM "3. PagedAttention CUDA Kernel Execution":
 *  one fused kernel reads the block table and stages the frames on chip, with no
 *  gathered copy of K/V in HBM.]
 *
 *   q             [S, H, D], row stride free (16-byte multiple), [H, D] contiguous.
 *   k_cache, v_cache  [num_blocks, B, H, D] contiguous, same dtype as q.
 *   block_tables  int32 [S, max_blocks], inner stride 1; row s lists the frames of
 *                 sequence s in logical order; entries past ceil(L_s/B) unread.
 *   context_lens  int32 [S], L_s = tokens attended (the newest appended included).
 *                 L_s == 0 gives a zero output row.
 *   scale         softmax scale, normally 1/sqrt(D).
 *   out           [S, H, D], same dtype as q, [H, D] contiguous.
 * Arithmetic: K/V/q converted to fp32, fp32 dot products, online softmax and
 * accumulation in fp32, one rounding to the output dtype.  Long contexts are
 * split into partitions processed by separate thread blocks and combined by the
 * log-sum-exp rule in the same kernel: the last partition of a (sequence, head) to
 * finish merges them.  Work is handed to a persistent
 * grid through an atomic counter.  Counter and split partials live in a
 * workspace the library owns: one per (device, stream), allocated (cudaMalloc)
 * and zeroed on the first call with that pair and grown on the first call that
 * needs more (keep such calls outside CUDA-graph capture), freed by
 * pa_shutdown().  Calls on one stream run in order; calls on different streams
 * use different workspaces.
 * Supported: dtype f32/f16/bf16; D in {64, 128, 256} (f32: {64, 128});
 * 1 <= B <= 256; max_blocks * B < 2^31, else PA_ERR_UNSUPPORTED.  Any S < 2^31:
 * every thread block keeps three int32 per sequence in shared memory beside its
 * staging ring, so a batch larger than one launch holds (about 13,000 sequences
 * with 4 heads of 128 fp16 per block) runs as launches over consecutive ranges of
 * sequences, one after another on the stream.
 * Bounded waits: every wait inside the kernels gives up after ~2 s, raising
 * PA_DEV_TIMEOUT (the outputs of that call are then undefined).  Reading the status
 * with pa_get_device_status marks this device's workspaces for re-zeroing, so later
 * calls start from clean counters; pa_shutdown() frees them outright.
 */
int pa_decode(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
              const pa_tensor* block_tables, const pa_tensor* context_lens,
              float scale, const pa_tensor* out, pa_stream stream);

/*
 * pa_prefill -- causal attention for chunks of queries (prefill / chunked
 * prefill) over the paged cache, on the tensor cores.
 * [MW "1. The Mathematical Foundation", the causal form o_i = sum_{j<=i}
 *  softmax(a_ij) v_j; "2. The Algorithmic Steps" (prompt tokens are written to the
 *  cache, then attention runs over the sequence's frames).]
 *
 *   q             [T, H, 128] fp16/bf16, row stride free (16-byte multiple).  Rows
 *                 query_start[s] .. query_start[s+1]-1 are the last
 *                 n_s = query_start[s+1] - query_start[s] positions of sequence s;
 *                 their K/V rows must already be in the cache (pa_cache_append).
 *   k_cache, v_cache  [num_blocks, B, H, 128], same dtype as q; B in {8, 16, 32, 64, 128}.
 *   block_tables  int32 [S, max_blocks]; context_lens int32 [S] = L_s (chunk included);
 *   query_start   int32 [S + 1], non-decreasing, query_start[S] <= T.
 *   out           [T, H, 128], same dtype; row r at position p = L_s - n_s + (r -
 *                 query_start[s]) gets sum_{j<=p} softmax(q_r . k_j * scale) v_j.
 * Arithmetic: q.k products accumulated in fp32 by the tensor cores, softmax in fp32,
 * the weights rounded to the cache dtype before the value product (fp32 accumulate),
 * normalisation in fp32.  Cache slots of a frame beyond L_s are read and must hold
 * finite values (the weights there are zero).  A sequence whose query range is not
 * inside [0, T] (query_start[s] < 0, query_start[s+1] < query_start[s] or > T), with
 * n_s > L_s or with L_s > max_blocks*B sets PA_DEV_BAD_LEN and its rows are left
 * untouched; ranges that overlap so much that they hold more 256-row tile pairs than
 * T rows allow set PA_DEV_BAD_LEN and nothing is computed.  Frame ids outside
 * [0, num_blocks) set PA_DEV_BAD_BLOCK and read as zeros.  Uses the (device, stream)
 * workspace's work counter; one thread block per SM; tile pairs are taken longest
 * first.  Every thread block keeps the tile-pair offsets and order of the batch in
 * shared memory (about 8000 entries, S + T/256 + 1 of them): a batch with more
 * sequences than that runs as launches over consecutive ranges of sequences (q and
 * out stay whole), one after another on the stream; PA_ERR_UNSUPPORTED only when T
 * alone leaves no room (T above about two million rows).
 */
int pa_prefill(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
               const pa_tensor* block_tables, const pa_tensor* context_lens,
               const pa_tensor* query_start, float scale, const pa_tensor* out,
               pa_stream stream);

/* ---- the split cache layout ["PagedAttention: Virtual Memory Guide for LLM
 * Inference", "3. PagedAttention CUDA Kernel Execution": the kernel signature stores
 * k_cache as [num_blocks, num_heads, head_dim/x, block_size, x] and v_cache as
 * [num_blocks, num_heads, head_dim, block_size], x = elements per 16 bytes].
 *
 * Same contract as pa_cache_append / pa_decode with the caches in that layout:
 * k_cache passed as the 4-D view [num_blocks, H, D/8, B*8] (each last-dim row holds
 * B chunks of 8 elements), v_cache as [num_blocks, H, D, B]; both contiguous, fp16 or
 * bf16, D in {64, 128}, B in {8, 16, 32}, H a multiple of 4 (else
 * PA_ERR_UNSUPPORTED).  pa_decode_split splits long contexts into partitions when the
 * (sequence, 4-head group) items cannot fill the GPU and then launches a second,
 * merging kernel; its partials use the (device, stream) workspace.  Status bits and
 * error codes as for pa_decode; as there, cache slots that hold no token of a sequence
 * may hold any bits (they never reach the result). */
int pa_cache_append_split(const pa_tensor* k_new, const pa_tensor* v_new, const pa_tensor* slot_mapping,
                          const pa_tensor* k_cache, const pa_tensor* v_cache, pa_stream stream);
int pa_decode_split(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                    const pa_tensor* block_tables, const pa_tensor* context_lens, float scale,
                    const pa_tensor* out, pa_stream stream);

/* Launch options for pa_decode_ex; 0 in any field = automatic choice. */
typedef struct pa_decode_params {
  int32_t partition_tokens;  /* >0: split context into partitions of this many tokens
                                (rounded up to a multiple of B); -1: never split */
  int32_t heads_per_cta;     /* 1, 2 or 4 (must divide H) */
  int32_t warps_per_head;    /* 1, 2, 4 or 8 */
  int32_t stages;            /* K/V staging buffers per thread block, 2..8 */
  int32_t ctas_per_sm;       /* persistent grid = SMs x this (clamped to occupancy) */
  int32_t items_per_cta;     /* 0 (default): keep whole sequences when they already give
                                every thread block work and the longest is at most the
                                average load per block, else aim at 1.5 work items per
                                thread block; >0: always aim at this many */
  int32_t generic_only;      /* 1: never take the unrolled full-frame path (testing) */
  int32_t share_prefix;      /* >0: read frames that consecutive sequences share once for
                                all of them (see below); 1 = runs of at least 256 shared
                                tokens, >1 = runs of at least this many tokens */
} pa_decode_params;

/* pa_decode with explicit launch options (tests, tuning).  params may be NULL.
 *
 * share_prefix > 0 -- shared-prefix decode.  The result is pa_decode's; only the
 * number of reads of shared frames changes.  Forks copy block tables and raise
 * reference counts ("PagedAttention: Virtual Memory Guide for LLM Inference", "Key
 * Architectural Mechanics"), so siblings' tables begin with the same frame ids, and
 * for the tokens in those frames their keys and values are the same bytes.  A first
 * kernel finds, for every sequence s >= 1, how many leading tokens it reads through
 * the same frame ids as sequence s-1 (equal leading table entries, capped by both
 * context lengths).  Runs of consecutive sequences whose count reaches the
 * threshold (share_prefix == 1: 256 tokens; > 1: that many; never below B) are cut
 * into chunks of up to 16; each chunk's smallest count, rounded down to whole
 * frames, is its shared prefix, attended once with all members' queries (one read of
 * each shared frame, the queries as the rows of a tensor-core tile), while each
 * member's remaining tokens are attended alone; the parts are merged by the
 * log-sum-exp rule.  Put sibling sequences next to each other in the batch to
 * benefit.  Arithmetic: q.k products and the weighted sums of values on the tensor
 * cores with fp32 accumulation, the weights carried as two 16-bit parts (fp32
 * accurate), softmax in fp32.  Applies to fp16 / bf16 caches with D = 128, B a power
 * of two >= 8 and 2 <= S <= 4096 (other shapes run the plain decode, with the same
 * result).  heads_per_cta, when given, must be 1, 2 or 4 and warps_per_head 0 or 1,
 * else PA_ERR_INVALID.  Uses workspace partials for every sequence that has more than
 * one part, and launches two kernels: the plan, then the decode, whose thread blocks
 * merge the split sequences by the log-sum-exp rule once they have no items left. */
int pa_decode_ex(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                 const pa_tensor* block_tables, const pa_tensor* context_lens,
                 float scale, const pa_tensor* out, const pa_decode_params* params,
                 pa_stream stream);

/*
 * pa_decode_static -- pa_decode that allocates nothing.  (No counterpart in the
 * pages: an addition for callers that cannot allocate device memory.)
 *
 * Who needs it: a process whose device memory is entirely owned by its own pool
 * allocator (a cudaMalloc from this library could fail or fragment that pool), or
 * a latency-bound loop that cannot take the device-wide synchronisation of a
 * first cudaMalloc.  pa_decode would allocate its workspace on first use; this
 * entry point instead uses a fixed 16 MiB scratch array compiled into the library
 * (a file-scope __device__ array that every GPU which loads the library keeps
 * until the process exits).
 *
 * Arguments, results and error checks are those of pa_decode with automatic
 * launch options; the caller still provides every input and output.
 *   - One launch only: PA_ERR_UNSUPPORTED when S is more than one launch holds
 *     (pa_decode would split the batch).
 *   - Returns PA_ERR_SCRATCH_LIMIT, launching nothing, when the problem needs more
 *     than 16 MiB of scratch: 256 B of work counters and, when a context may be
 *     split, S*H int32 arrival counters plus room for up to
 *     (3 * resident thread blocks + S*H/heads_per_cta) partial results of
 *     heads_per_cta*(head_dim + 2) floats each (about 6 MiB for 64 sequences of up
 *     to 2048 tokens with 32 heads of 128).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call before
 *     any stream capture.
 *   - Every call shares the one array and each call zeroes its counters with
 *     cudaMemsetAsync on `stream` before the kernels: calls whose kernels overlap on
 *     the GPU (different streams, or other threads) race on it.  Serialise them.
 */
int pa_decode_static(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                     const pa_tensor* block_tables, const pa_tensor* context_lens,
                     float scale, const pa_tensor* out, pa_stream stream);

/* Synchronises `stream` (and then the device), returns the current device's sticky
 * PA_DEV_* bits in *status_out and clears them.  When PA_DEV_TIMEOUT was set, the
 * scheduler and arrival counters of every workspace of this device are re-zeroed on
 * their next use (a block that gave up may have left them non-zero). */
int pa_get_device_status(pa_stream stream, int32_t* status_out);

/* Human-readable name of a return code (static storage). */
const char* pa_strerror(int code);

/* Number of kernels this library has launched in this process (all devices). */
int64_t pa_launch_count(void);

/* Frees the library-owned decode workspaces of every device.  Call only when no
 * decode launched by this library is still running. */
int pa_shutdown(void);

/* ===================================================================================
 * Host block manager (pure host code; no GPU needed)
 * [VM "Reference Implementation: Block Table & Paged Cache Manager",
 *  "Key Architectural Mechanics / 1-2"; MW "Implementation", BlockManager;
 *  SE "How PagedAttention solves it"]
 * Free frames leave from the front of the free list and return to its back when
 * their reference count reaches zero.  Sequences are named by caller-chosen
 * int64 ids.  Not thread-safe: one handle per thread, or external locking.
 * =================================================================================== */
typedef struct pa_bm pa_bm;

/* free_order: NULL = 0,1,...,num_blocks-1; else a permutation of those ids that
 * becomes the initial free list.  num_blocks * block_size must fit in int32. */
int  pa_bm_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order,
                  pa_bm** bm_out);
void pa_bm_destroy(pa_bm* bm);

/* New sequence with a prompt of num_tokens: takes ceil(num_tokens/B) frames,
 * all-or-nothing [MW BlockManager.allocate].  slots_out (nullable) receives the
 * num_tokens flat slots of the prompt tokens. */
int pa_bm_add_seq(pa_bm* bm, int64_t seq_id, int32_t num_tokens, int32_t* slots_out);

/* One new token for seq_id [VM "1. Demand Paging", "2. Copy-on-Write"]:
 *   t = current length; if t % B == 0 a frame is taken from the free list and
 *   appended to the table; else if the tail frame is shared (refcount > 1) a
 *   private frame is taken, the shared frame loses one reference and the private
 *   one replaces it in the table; the caller must then copy the frame's data
 *   (*cow_src -> *cow_dst, both -1 when there is nothing to copy).
 *   *slot_out = flat slot of token t.  All-or-nothing. */
int pa_bm_append(pa_bm* bm, int64_t seq_id, int32_t* slot_out,
                 int32_t* cow_src, int32_t* cow_dst);

/* One decode step: pa_bm_append for seq_ids[0..n) in that order, all-or-nothing
 * (if any append would run out of frames or names an unknown sequence, nothing
 * changes).  slots_out [n]; copies_out [n][2] receives the (src, dst) pairs in
 * issue order, *n_copies_out their count. */
int pa_bm_step(pa_bm* bm, const int64_t* seq_ids, int32_t n, int32_t* slots_out,
               int32_t* copies_out, int32_t* n_copies_out);

/* A prompt chunk: num_tokens new tokens for one sequence, each following the
 * pa_bm_append rule in turn, all-or-nothing.  slots_out [num_tokens]; copies_out
 * (nullable) [num_tokens][2] receives copy-on-write pairs (at most one, for the
 * first token), *n_copies_out their count (nullable). */
int pa_bm_extend(pa_bm* bm, int64_t seq_id, int32_t num_tokens, int32_t* slots_out,
                 int32_t* copies_out, int32_t* n_copies_out);

/* ---- prefix caching ["PagedAttention: Virtual Memory Guide for LLM Inference",
 * "2. Native Synergy with RadixAttention and Prompt Caching": filled blocks are
 * immutable, so a prompt whose token prefix is already in the cache maps those
 * blocks onto the frames holding them, with no recomputation].
 *
 * A filled block of a sequence admitted with token ids is registered under the key
 * (node of the block before it, its B token ids); nodes form a trie and their ids
 * are never reused.  A freed frame keeps its block registered and goes to the back
 * of the free list as usual; the registration is dropped (evicted) only when the
 * free list hands the frame out again.  Sequences admitted without token ids, and
 * their forks, never register blocks; an append without a token id leaves its
 * block (and every later block of that sequence) unregistered.
 *
 * pa_bm_add_seq_cached: admit a prompt of num_tokens token ids [num_tokens].  Its
 * leading filled blocks that are registered (looked up in order, stopping at the
 * first miss; a block holding the prompt's last token never counts) are shared:
 * each gains a reference, leaving the free list if it was there.  The remaining
 * blocks come from the free list (blocks filled by the prompt are registered; if
 * the same content is registered already the existing node stands for it).
 * *n_cached_out = tokens found in the cache (a multiple of B, < num_tokens unless
 * num_tokens is 0); slots_out [num_tokens] receives the slots of tokens
 * n_cached .. num_tokens-1, whose K/V rows the caller must write.  All-or-nothing:
 * PA_ERR_OUT_OF_BLOCKS (counting cached frames about to be reused as taken) leaves
 * every state unchanged; PA_ERR_SEQ_EXISTS for a live id.
 * pa_bm_step_tokens / pa_bm_extend_tokens: pa_bm_step / pa_bm_extend with the id of
 * each appended token (tokens [n]), so that blocks they fill are registered.
 * pa_bm_cached_frames: out[f] = 1 if frame f holds a registered block (out may be
 * NULL when cap is 0); *n_cached_out = how many do. */
int pa_bm_add_seq_cached(pa_bm* bm, int64_t seq_id, const int32_t* tokens, int32_t num_tokens,
                         int32_t* slots_out, int32_t* n_cached_out);
int pa_bm_step_tokens(pa_bm* bm, const int64_t* seq_ids, const int32_t* tokens, int32_t n,
                      int32_t* slots_out, int32_t* copies_out, int32_t* n_copies_out);
int pa_bm_extend_tokens(pa_bm* bm, int64_t seq_id, const int32_t* tokens, int32_t num_tokens,
                        int32_t* slots_out, int32_t* copies_out, int32_t* n_copies_out);
int pa_bm_cached_frames(const pa_bm* bm, int32_t* out, int32_t cap, int32_t* n_cached_out);

/* Zero-copy fork: child shares every frame of parent (each gains a reference)
 * and inherits its length [VM "2. Zero-Copy Branching"]. */
int pa_bm_fork(pa_bm* bm, int64_t parent_id, int64_t child_id);

/* Release a finished sequence: each frame loses a reference, in table order;
 * frames reaching zero return to the back of the free list.  An id that is not
 * live is a no-op returning PA_WARN_DOUBLE_FREE. */
int pa_bm_free(pa_bm* bm, int64_t seq_id);

/* Batched forms for a search step (beam search keeps the survivors' forks and drops
 * the rest in one call each).  pa_bm_fork_many performs n forks in order, all or
 * nothing: the whole batch is checked first (a child forked earlier in the batch may
 * be a later parent); PA_ERR_UNKNOWN_SEQ / PA_ERR_SEQ_EXISTS leave the manager
 * unchanged.  pa_bm_free_many frees in order exactly as n pa_bm_free calls would and
 * returns PA_WARN_DOUBLE_FREE if any id was not live (the others are still freed). */
int pa_bm_fork_many(pa_bm* bm, const int64_t* parent_ids, const int64_t* child_ids, int32_t n);
int pa_bm_free_many(pa_bm* bm, const int64_t* seq_ids, int32_t n);

/* One decode step of a batch with the host side done natively: pa_bm_step for
 * seq_ids[0..n) (one token each, copy-on-write as pa_bm_append), the batch's slots,
 * block tables [n, max_blocks] and lengths staged in a library-owned ring of mapped
 * pinned host memory (per device and stream, four slots, each reused only after the
 * kernel that last read it has run), then pa_copy_blocks (when a shared tail was
 * written), pa_cache_append of k_new / v_new [n, H, D] (device) at the step's slots,
 * and pa_decode_ex of q [n, H, D] into out, all on `stream`.  The frame copies of a
 * step (up to 256 of them) carry their (src, dst) pairs in the copy kernel's launch
 * parameters; the append reads its slots from the ring directly and copies the
 * tables and lengths to device memory in the same launch.  A step with more than 256
 * copies uploads the staged block with one asynchronous copy first and runs
 * pa_copy_blocks on the device pairs.  params may be NULL:
 * automatic launch options, with share_prefix = 1 when auto_share is set and two
 * neighbouring sequences of the batch start on the same frame.  *n_copies_out (may
 * be NULL) receives the number of frame copies; lens_out (host, n entries, may be
 * NULL) the context lengths attended.  Errors: those of pa_bm_step leave everything
 * unchanged and launch nothing; PA_ERR_CAPACITY (a table longer than max_blocks) and
 * errors of the device calls come after the block-manager step, which stands. */
int pa_step_decode(pa_bm* bm, const int64_t* seq_ids, int32_t n, int32_t max_blocks,
                   const pa_tensor* k_new, const pa_tensor* v_new, const pa_tensor* q,
                   const pa_tensor* k_cache, const pa_tensor* v_cache, float scale,
                   const pa_tensor* out, const pa_decode_params* params, int32_t auto_share,
                   pa_stream stream, int32_t* n_copies_out, int32_t* lens_out);

/* Block tables [n, max_blocks] (row-major, unused entries -1) and lengths [n] of
 * the listed sequences, ready to upload for pa_decode.  PA_ERR_CAPACITY if a
 * table is longer than max_blocks. lens_out may be NULL. */
int pa_bm_block_tables(const pa_bm* bm, const int64_t* seq_ids, int32_t n,
                       int32_t max_blocks, int32_t* tables_out, int32_t* lens_out);

/* Queries. */
int pa_bm_seq_info(const pa_bm* bm, int64_t seq_id, int32_t* len_out, int32_t* n_blocks_out);
int pa_bm_table(const pa_bm* bm, int64_t seq_id, int32_t* out, int32_t cap, int32_t* n_out);
int pa_bm_slot(const pa_bm* bm, int64_t seq_id, int32_t pos, int32_t* slot_out);
int pa_bm_num_free(const pa_bm* bm, int32_t* n_out);
int pa_bm_free_list(const pa_bm* bm, int32_t* out, int32_t cap, int32_t* n_out);  /* front first */
int pa_bm_ref_counts(const pa_bm* bm, int32_t* out, int32_t cap);               /* [num_blocks] */
int pa_bm_num_seqs(const pa_bm* bm, int32_t* n_out);

/* Self-test of the failure path of every kernel's bounded waits (each mbarrier wait
 * gives up after ~2 s at the maximum SM clock, raises PA_DEV_TIMEOUT in the status
 * word and makes the thread block's later waits return at once, so a stuck copy ends
 * the kernel with an error instead of hanging the GPU).  Launches one small kernel on
 * `stream` whose first warp waits on an mbarrier that nothing arrives on, then whose
 * second warp waits on the same barrier; synchronises the stream and writes
 * result_out[4] (host): the two waits' results (1 = completed, 0 = gave up) and the SM
 * cycles each took.  Expected: {0, 0, > 4e9, small}, and PA_DEV_TIMEOUT set for the
 * next pa_get_device_status.  Takes about two seconds; the context stays usable.
 * Errors: PA_ERR_INVALID (result_out NULL), PA_ERR_CUDA. */
int pa_selftest_wait_timeout(int64_t* result_out, pa_stream stream);

/* Snapshot of the whole manager into caller buffers (parity checks against a reference
 * manager, debugging, inspection), the state the "Reference Implementation" of
 * "PagedAttention: Virtual Memory Guide for LLM Inference" keeps: the live sequences in
 * ascending id order -- ids_out[n_seqs], lens_out[n_seqs], table_offsets_out[n_seqs + 1]
 * (table of sequence i = tables_out[table_offsets_out[i] .. table_offsets_out[i+1])) --,
 * the free list front first (free_out[n_free]) and every frame's reference count
 * (refs_out[num_blocks]).  cap_seqs bounds ids_out / lens_out (table_offsets_out holds
 * cap_seqs + 1), cap_entries bounds tables_out; free_out and refs_out must hold
 * num_blocks entries.  The sizes needed are written to *n_seqs_out, *n_entries_out and
 * *n_free_out (each may be NULL) even when a buffer is too small, which returns
 * PA_ERR_CAPACITY and writes nothing else.  Read only.  PA_ERR_INVALID for a NULL
 * manager or output buffer, or negative capacities. */
int pa_bm_export(const pa_bm* bm, int64_t* ids_out, int32_t* lens_out, int64_t* table_offsets_out,
                 int32_t* tables_out, int32_t* free_out, int32_t* refs_out, int32_t cap_seqs,
                 int64_t cap_entries, int32_t* n_seqs_out, int64_t* n_entries_out, int32_t* n_free_out);

/* Memory accounting of the pool as it stands.  Pages: "PagedAttention: Virtual
 * Memory Guide for LLM Inference", "The Solution" (frames are granted on demand, so
 * a sequence wastes only the unfilled slots of its last frame: fewer than B) and
 * "2. Zero-Copy Branching via Copy-on-Write" (forked sequences hold shared frames
 * once); "Solving the LLM Memory Wall", "Performance Analysis" (slots allocated
 * against tokens held).  Fields, all counts:
 *   num_seqs        live sequences
 *   frames_total    frames in the pool (num_blocks)
 *   frames_in_use   frames with a reference count above zero
 *   frames_cached   free frames that still hold a registered block of the prefix
 *                   cache (reusable by a prompt with the same token prefix)
 *   table_entries   sum of the live sequences' table lengths: the frames they would
 *                   hold without sharing
 *   tokens_logical  sum of the live sequences' lengths
 *   slots_filled    token slots of frames in use that hold a token of a live
 *                   sequence; a frame counts the largest fill any of its sharers
 *                   gives it (sequence length minus the frame's first position,
 *                   clamped to [0, B])
 *   max_seq_waste   largest (table length * B - length) over live sequences, 0 when
 *                   there are none; always < B
 * Derived: paged waste = 1 - slots_filled / (frames_in_use * B); saving from shared
 * frames = 1 - frames_in_use / table_entries.  Read only; O(num_blocks + total table
 * length) time.  Errors: PA_ERR_INVALID for a NULL argument. */
typedef struct {
  int64_t num_seqs;
  int64_t frames_total;
  int64_t frames_in_use;
  int64_t frames_cached;
  int64_t table_entries;
  int64_t tokens_logical;
  int64_t slots_filled;
  int64_t max_seq_waste;
} pa_bm_usage_t;
int pa_bm_usage(const pa_bm* bm, pa_bm_usage_t* out);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* PA_H_ */
