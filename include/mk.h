/*
 * mk.h -- C ABI of the persistent decode megakernel for GB300 (sm_103a).
 *
 * One decode step of a whole Llama-style decoder runs as ONE resident kernel launch: a grid of
 * S CTAs (one per SM) in which every CTA interprets its own queue of tile instructions, waits
 * for an instruction's inputs (epoch-tagged data, or global completion counters: mk_set_sync),
 * streams the instruction's weights / KV rows through leased shared-memory pages, runs the
 * operator body and publishes its completions.
 * The design follows the "Inference MegaKernel" page, section "Hand-written whole-model
 * MegaKernel" (principle, scheduling and data flow; its control-flow pseudocode; its object
 * table), and the four device-protocol contracts of its section "Unified framework" (data
 * visibility, forward progress, capacity, resources).
 *
 * Conventions
 *  - Every call returns an mk_status; nothing aborts or throws across the ABI.  After a non-OK
 *    status mk_last_error() holds a message (thread-local).
 *  - All device memory of the model (weights, KV cache, completion counters, scratch, logits)
 *    is allocated and owned by the caller; the library only borrows the pointers for the
 *    lifetime of the bound context.  The library owns its host schedule objects and, per bound
 *    context, one small device copy of the queues, counter totals and layer pointer table.
 *  - Weights and KV cache are bf16, row-major, every pointer 16-byte aligned.
 *  - "pos" is the position the step's token occupies; the step appends its K/V at pos and
 *    attends over positions 0..pos inclusive.
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MK_OK = 0,
    MK_ERR_ARG = 1,        /* a bad argument (null, misaligned, out of range, unsupported shape) */
    MK_ERR_CAPACITY = 2,   /* queue / page ring / KV capacity cannot hold the configuration     */
    MK_ERR_RESOURCES = 3,  /* the kernel cannot be made resident with one CTA on S SMs          */
    MK_ERR_CUDA = 4,       /* a CUDA runtime call failed                                        */
    MK_ERR_TIMEOUT = 5,    /* a device wait ran out its time budget (the step was abandoned)    */
    MK_ERR_OPCODE = 6,     /* the device met an invalid opcode in a queue                       */
    MK_ERR_BOUNDS = 7,     /* the device met an instruction whose fields are out of range       */
    MK_ERR_POISONED = 8    /* an earlier device error poisoned this context; unbind and re-bind */
} mk_status;

/* Model configuration (a Llama-style decoder).  batch <= 8; n_q_heads % n_kv_heads == 0 with
 * at most 8 query heads per KV head; head_dim a multiple of 16 and <= 128; hidden, ffn and
 * n_q_heads * head_dim multiples of 8 and <= 16384. */
typedef struct {
    int32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
    int32_t tied_embeddings; /* informational: the LM head pointer may equal the embedding  */
    int32_t batch;           /* sequences decoded together in one step                      */
    int32_t max_seq;         /* KV capacity in positions; every pos must be < max_seq       */
    double rms_eps, rope_theta;
} mk_model_cfg;

/* Schedule knobs; pass NULL to mk_build_schedule for the defaults (each 0 field = default).
 * With tile_bytes 0 every matvec operator is cut into about sm_count tiles (QKV tiles at most
 * head_dim rows), each streamed through the page ring page by page (at batch > 1 a tile whose rows
 * are longer than 2048 takes at most 64 rows: its sums stay in registers over the staging
 * ranges); otherwise tiles hold about tile_bytes.  A row's arithmetic never depends on the
 * tiling.
 * kv_limit is the variable-length re-planning of the page's boundaries paragraph ("Inference
 * MegaKernel", section "Hand-written whole-model MegaKernel": dynamic batches and variable-length
 * requests change the static queue): attention chunks past a sequence's window get no tile, so a
 * batch of uneven lengths is placed by the work it has; mk_rebind_schedule moves a binding to a
 * schedule with new windows. */
typedef struct {
    int32_t page_bytes;  /* shared-memory page size (a power of two); default 32768, at batch > 1
                            65536 (a page is then a 16-row block over page_bytes / 32 positions,
                            which must divide the 2048-position staging range: MK_ERR_ARG) */
    int32_t tile_bytes;  /* 0: per-SM tiles (see above); else the target weight bytes per matvec
                            tile (capped at 8 rows for QKV, O and down, 16 gate/up pairs, 32
                            LM-head rows)                                                        */
    int32_t attn_chunk;  /* KV positions per split-K attention tile; 0: 128, doubled (up to 512)
                            while batch * n_kv_heads * ceil(max_seq / chunk) > 152 (a property
                            of the configuration, not of sm_count)                               */
    int32_t rows_qkv, rows_o, pairs_up, rows_down, rows_lm; /* explicit rows (pairs) per tile,
                            overriding the above; rows_qkv <= head_dim                           */
    uint64_t shuffle_seed; /* 0: cost-ordered placement; otherwise a seeded shuffled placement  */
    int32_t kv_limit[8];   /* per sequence: positions the schedule serves, [0, kv_limit) (0 or
                            max_seq: all); a step at pos >= kv_limit[b] is rejected (MK_ERR_ARG) */
} mk_sched_opts;

typedef struct mk_schedule mk_schedule; /* opaque, library-owned host object */
typedef struct mk_ctx mk_ctx;           /* opaque, library-owned bound context */

/* Host scheduler (page section "Hand-written whole-model MegaKernel": cut every operator into
 * tiles, build the tile dependency DAG, assign waves and a memory/compute pool, place tiles on
 * the SMs' instruction queues, tensorise each queue as [S, Q, 32] int32).
 * Tiles: per layer QKV rows (RMSNorm prologue), split-K attention chunks (RoPE + KV append in
 * the chunk that holds pos; the chunk that completes its KV group also does the group's
 * log-sum-exp combine), O rows (+ residual), gate/up row pairs (SiLU(gate)*up), down rows
 * (+ residual; at batch > 1 with ffn > 2048 one tile per (2048-position staging range, row
 * block), the last range's tile adding the others' partial sums); then LM-head rows (final
 * RMSNorm prologue, running max/argmax) and one argmax per sequence.
 * sm_count: number of queues (= CTAs launched), 1 <= sm_count <= 4096.
 * opts: NULL for defaults.  On success *out receives a new schedule (free with
 * mk_schedule_free).  Errors: MK_ERR_ARG (bad cfg/opts), MK_ERR_CAPACITY (a tile needs more
 * than 2^20 bytes of pages, or the model exceeds the encoding's ranges). */
mk_status mk_build_schedule(const mk_model_cfg* cfg, int32_t sm_count, const mk_sched_opts* opts,
                            mk_schedule** out);

/* The queues: a read-only pointer to S*Q*32 int32 (row-major [S, Q, 32]) valid until the
 * schedule is freed.  The page's object table ("Inference MegaKernel", section "Hand-written
 * whole-model MegaKernel") lists the instruction queue as an int32 tensor of shape [S, Q, 32]
 * held in HBM for the life of the kernel; the word layout is this library's (the page gives none).
 * Errors: MK_ERR_ARG on a null argument.  Word layout of one instruction:
 *   [0] opcode (0 END, 1 QKV, 2 ATTN, 3 COMB, 4 OPROJ, 5 UPGATE, 6 DOWN, 7 LMHEAD, 8 ARGMAX;
 *       COMB, the combine of one (sequence, KV group)'s chunk partials, exists at batch > 1 only)
 *   [1] layer (n_layers for LMHEAD / ARGMAX)   [2] sequence b (attention, combine, argmax)
 *   [3] a0: first row | KV group             [4] a1: rows (pairs for UPGATE) | chunk | #LM tiles
 *   [5] a2: chunk length (ATTN, COMB) | LM tile index (LMHEAD) | staging range (DOWN at batch
 *       > 1 with ffn > 2048: the tile covers positions [2048 a2, 2048 (a2 + 1)) of its rows; a
 *       tile of a lower range completes nothing and stores its partial sums, the tile of the
 *       last range, of a higher id in the same wave, waits for them, adds them in range order,
 *       writes the rows and completes)
 *   [6] number of waits (<= 4)   [7..14] (counter, need) pairs
 *   [15] number of completions (<= 2)   [16..19] (counter, delta) pairs
 *   [20] pages of the largest stream the tile may need   [21] tile id   [22] wave
 *   [23] 1 = conditional completions (ATTN at batch 1): only the tile whose chunk holds the
 *        step's position fires them; it combines the group's chunk partials, waiting inside its
 *        wave for the lower chunks (each queue runs its tiles of a wave in tile-id order).  At
 *        batch > 1 it is 0: the chunk tiles complete nothing and the group's COMB tile, of a
 *        higher id in the same wave, waits for their partials, combines them and completes
 *   [24..31] 0 (the bound device copy carries the tile's resolved stream addresses in [26..31])
 * A wait is satisfied when counter - (epoch * total[counter] + need) >= 0 (mod 2^32).  END is
 * all zeros and pads every queue. */
mk_status mk_schedule_queues(const mk_schedule* s, const int32_t** queues, int32_t* sm_count,
                             int32_t* queue_len);

/* Per-step counter totals: total[c] = sum of the deltas published into counter c in one step
 * (read-only pointer to n uint32, valid until the schedule is freed).  The page's object table
 * lists global completion counters beside the queues; its interpreter waits until a counter has
 * reached what an instruction needs and adds to the counters an instruction completes (section
 * "Hand-written whole-model MegaKernel", pseudocode and object table).  With counters that keep
 * growing across steps the wait target is epoch * total + need.  Errors: MK_ERR_ARG on a null
 * argument. */
mk_status mk_schedule_counters(const mk_schedule* s, const uint32_t** totals, int32_t* n_counters);

/* The schedule's attention chunk (KV positions per split-K attention tile: the option, or the
 * default the scheduler chose); a paged KV cache must use it as its block size.  MK_ERR_ARG on
 * null arguments. */
mk_status mk_schedule_attn_chunk(const mk_schedule* s, int32_t* out);

/* Overwrites one word of the host queue copy (for fault-injection tests of the device runtime's
 * checks; contexts bound earlier are not affected).  MK_ERR_ARG if an index is out of range. */
mk_status mk_schedule_patch(mk_schedule* s, int32_t sm, int32_t slot, int32_t word, int32_t value);

/* Bytes of device scratch a context of this schedule needs (activations, attention partials,
 * LM-head partials, RoPE table, error word, output tokens) -- the activation objects the page's
 * object table keeps in HBM for the resident execution (section "Hand-written whole-model
 * MegaKernel").  The caller allocates them (mk_bind).  0 if s is NULL. */
size_t mk_scratch_bytes(const mk_schedule* s);

void mk_schedule_free(mk_schedule* s);

/* Device weights, bf16 row-major, caller-owned.  Per-layer fields are HOST arrays of n_layers
 * DEVICE pointers (copied at bind).  Layouts:
 *   embed      [vocab, hidden]
 *   lm_head    [vocab, hidden]          (may equal embed when tied)
 *   final_norm, attn_norm[l], mlp_norm[l]   [hidden]
 *   wqkv[l]    [(n_q_heads + 2 n_kv_heads) head_dim, hidden]   rows: q heads, k heads, v heads
 *   wo[l]      [hidden, n_q_heads head_dim]
 *   wgate_up[l][2 ffn, hidden]          rows: gate rows, then up rows
 *   wdown[l]   [hidden, ffn] */
typedef struct {
    const void* embed;
    const void* lm_head;
    const void* final_norm;
    const void* const* attn_norm;
    const void* const* wqkv;
    const void* const* wo;
    const void* const* mlp_norm;
    const void* const* wgate_up;
    const void* const* wdown;
} mk_weights;

/* KV cache, bf16, caller-owned (the page's object table lists the K/V cache as a per-layer
 * object in HBM that lives as long as the request).
 * Element (b, l, g, p, e) of K lives at k + b*batch_stride + l*layer_stride + g*head_stride
 * + p*head_dim + e (strides in elements, each a multiple of 8); V likewise. */
typedef struct {
    void* k;
    void* v;
    int64_t batch_stride, layer_stride, head_stride;
} mk_kv;

/* Paged KV cache (optional, see mk_bind_paged).  The K (and V) cache is a pool of blocks of
 * block_size positions per (layer, KV head); sequence b's positions [j*block_size,
 * (j+1)*block_size) live in pool block block_table[b*max_blocks + j].  Element (b, l, g, p, e) of
 * K lives at k + l*layer_stride + g*head_stride + (block_table[b*max_blocks + p/block_size]*
 * block_size + p % block_size)*head_dim + e (mk_kv's batch_stride is not used).  The page calls
 * the KV cache paged and per layer; one block is one split-K attention chunk, so a chunk's rows
 * are one contiguous copy.
 *  block_table  DEVICE int32[batch * max_blocks], caller-owned, 4-byte aligned; read by every
 *               step (the caller may rewrite it between steps).  An entry outside [0, n_blocks)
 *               that a step needs stops the step with MK_ERR_BOUNDS (nothing is accessed there).
 *  block_size   positions per block: must equal the schedule's attention chunk
 *               (mk_schedule_attn_chunk).
 *  max_blocks   table entries per sequence, max_blocks * block_size >= max_seq.
 *  n_blocks     blocks in the pool per (layer, KV head): head_stride >= n_blocks*block_size*head_dim. */
typedef struct {
    const int32_t* block_table;
    int32_t block_size, max_blocks, n_blocks;
} mk_kv_pages;

/* Binds a schedule to one model instance on the current CUDA device (the page's model binding:
 * weights, KV cache, activations and counters become objects of the one resident execution,
 * bound once).
 * counters: device uint32[n_counters], caller-owned; zeroed by mk_bind.
 * scratch:  device buffer of >= mk_scratch_bytes(s) bytes, 256-byte aligned, caller-owned.
 * stream:   a cudaStream_t (NULL = legacy default stream); every launch of the context goes on it.
 * Checks shapes against the configuration, pointer alignment, that the largest tile fits the
 * shared-memory page ring (capacity contract) and that one CTA per SM can be resident with the
 * kernel's registers and shared memory (resources contract).  The schedule may be freed after
 * binding.  Errors: MK_ERR_ARG, MK_ERR_CAPACITY, MK_ERR_RESOURCES, MK_ERR_CUDA. */
mk_status mk_bind(const mk_schedule* s, const mk_weights* w, const mk_kv* kv, uint32_t* counters,
                  void* scratch, void* stream, mk_ctx** out);

/* mk_bind with a paged KV cache (pages non-NULL; NULL binds the contiguous layout exactly as
 * mk_bind).  Errors as mk_bind, plus MK_ERR_ARG for a block size other than the schedule's
 * attention chunk, a table that cannot cover max_seq, or strides that do not cover the pool. */
mk_status mk_bind_paged(const mk_schedule* s, const mk_weights* w, const mk_kv* kv, const mk_kv_pages* pages,
                        uint32_t* counters, void* scratch, void* stream, mk_ctx** out);

/* Moves a binding to another schedule of the same model configuration, SM count, page size,
 * attention chunk and tile rows -- in practice one built with other kv_limit windows (the
 * re-planning for a changing batch of variable-length requests; see mk_sched_opts).  The new
 * queues are resolved against the bound weights and uploaded; counters, epoch, KV cache and
 * scratch carry over, so decoding continues where it was.  Waits for the bound stream first.
 * Errors: MK_ERR_ARG (null argument, an incompatible schedule, a persistent launch in flight),
 * MK_ERR_POISONED, MK_ERR_CUDA. */
mk_status mk_rebind_schedule(mk_ctx* c, const mk_schedule* s);

/* Time budget, in nanoseconds, of a single device wait: counter spins and tagged-data polls get
 * ns, waits of the consumer warps on one another 2 ns, the loader's and publisher's waits (which
 * only follow the consumers) 4 ns -- so the wait nearest the cause of a stall is the one recorded.
 * When one runs out the kernel records MK_ERR_TIMEOUT, every CTA leaves its loop after draining
 * its copies in flight, and the context is poisoned.  Default 2e9 (2 s). */
mk_status mk_set_timeout(mk_ctx* c, uint64_t ns);

/* How a consumer learns that the inputs of its instruction are ready.
 *  MK_SYNC_TAGS (default): the activation vectors one operator hands to the next (q/k/v,
 *    attention output, both residual streams, SwiGLU output) are tagged and a consumer polls
 *    the elements it reads until each carries this step's tag: q/k/v (and the attention chunk
 *    partials) as 64-bit words holding the fp32 value and the step's tag; the SwiGLU output,
 *    the residual streams and the attention output (every SM reads them whole) as 32-bit fp32
 *    words whose three low mantissa bits hold a 3-bit step tag.  One read
 *    both proves readiness and fetches the data, so a dependency costs one memory round trip
 *    instead of the publisher's release fence, the counter add, the consumer's counter poll and
 *    then the data read.  Such a consumer reads no counter at all.  Counters are still
 *    published, and they keep acquire/release semantics where a reader has no tag to check (the
 *    argmax over the LM-head partials, matvec inputs of 64-bit words cut into segments).
 *  MK_SYNC_COUNTERS: every instruction first waits all of its counters with acquire semantics
 *    (the page's protocol: wait the counters, run the body, fence, then add the completions);
 *    the tag checks then pass at the first read.
 * Both modes run the same arithmetic in the same order: their results are bit-identical.
 * Takes effect at the next launch.  Errors: MK_ERR_ARG (null context, unknown mode). */
typedef enum { MK_SYNC_TAGS = 0, MK_SYNC_COUNTERS = 1 } mk_sync_mode;
mk_status mk_set_sync(mk_ctx* c, int32_t mode);

/* Per-instruction timeline for profiling (the page's scheduling ledger: scheduler cycles,
 * dependency waits).  buf: DEVICE uint64[S * Q * 8] (caller-owned) or NULL to switch tracing off.
 * While on, every launch writes globaltimer stamps (ns) for instruction (sm, slot) at
 * buf[(sm * Q + slot) * 8 + k]: k = 0 slot published by the loader, 1 its pages issued,
 * 2 dependencies satisfied, 3 body done, 4 completions published, 6 (matvec) input vector
 * loaded, 7 (matvec) rows done -- 2, 3, 6 and 7 as seen by consumer warp 0;
 * buf[sm * Q * 8 + 5] = CTA start.  Entries of slots a CTA never reached keep their old
 * contents. */
mk_status mk_set_trace(mk_ctx* c, uint64_t* buf);

/* One decode step, synchronous -- the step the page's megakernel runs as one resident execution
 * per token (section "Hand-written whole-model MegaKernel": the whole decode step of the model
 * in one launch, instead of about a hundred kernels; section "Why inference still has
 * bubbles" for the launch and tail costs it removes).  tokens and pos are HOST arrays of `batch`
 * int32; logits is a DEVICE fp32 buffer [batch, vocab] (caller-owned) that receives the step's
 * logits;
 * next_tokens is a HOST array of `batch` int32 that receives the greedy (argmax, lowest index
 * on ties) next tokens.  Launches the resident grid once on the bound stream, then waits for it.
 * Errors: MK_ERR_ARG (token or pos out of range), MK_ERR_POISONED, MK_ERR_TIMEOUT,
 * MK_ERR_OPCODE, MK_ERR_BOUNDS (device-detected; they poison the context), MK_ERR_CUDA. */
mk_status mk_decode_step(mk_ctx* c, const int32_t* tokens, const int32_t* pos, float* logits,
                         int32_t* next_tokens);

/* One decode step like mk_decode_step, for callers that cannot allocate device memory: code
 * under a framework whose caching allocator owns the GPU's memory, or a latency-critical loop
 * where cudaMalloc / cudaFree may synchronise the device.  (The page has no counterpart: this is
 * an interface convenience of this library.)  Allocates nothing.  Instead of the scratch bound
 * with the context it uses one library-owned device array of MK_STATIC_SCRATCH_BYTES (16 MiB),
 * which every GPU that loads the library holds until the process exits.
 *  - The first call on a device sets the array up for that device (looks up its device
 *    address); make that first call before any stream capture.
 *  - A step that needs more scratch than the array holds is rejected with MK_ERR_CAPACITY
 *    (e.g. long contexts, whose attention partials grow with max_seq).
 *  - Every call shares the array and finds the previous call's contents; the call resets what
 *    must start fresh.  Calls that overlap on the GPU (other streams, other contexts at the same
 *    time) race on the array.
 * Arguments, results and errors as mk_decode_step (the context's counters and stream are used;
 * its bound scratch is not touched). */
#define MK_STATIC_SCRATCH_BYTES (16u << 20)
mk_status mk_decode_step_static(mk_ctx* c, const int32_t* tokens, const int32_t* pos, float* logits,
                                int32_t* next_tokens);

/* n_steps greedy decode steps in one call, each step's token fed to the next step's embedding on
 * the device (the chained, multi-step form of decoding, one launch per step; mk_decode_persistent
 * below runs all the steps in one launch).  Step i (0-based) decodes sequence b at position
 * pos[b] + i; step 0 takes tokens[b] (host), step i > 0 the greedy token of step i - 1.  The
 * steps are launched back to back on the bound stream, one launch each, with no host round trip
 * in between; the host synchronises once, at the end.
 *  tokens, pos   HOST int32[batch]: the first step's tokens (in [0, vocab)) and positions
 *                (pos[b] + n_steps <= max_seq).
 *  n_steps       >= 1.
 *  logits        DEVICE fp32[batch, vocab], caller-owned: every step writes it; the last step's
 *                logits remain.
 *  tokens_dev    DEVICE int32[n_steps * batch], caller-owned, 4-byte aligned: step i's greedy
 *                tokens at [i * batch, (i + 1) * batch).
 *  tokens_out    HOST int32[n_steps * batch]: a copy of tokens_dev, read back once at the end.
 * Errors: MK_ERR_ARG (null or misaligned pointer, n_steps < 1, a token or position out of range:
 * nothing is launched), MK_ERR_POISONED; a device error in any step is reported as by
 * mk_decode_step and poisons the context (later steps then stop at their first wait). */
mk_status mk_decode_steps(mk_ctx* c, const int32_t* tokens, const int32_t* pos, int32_t n_steps, float* logits,
                          int32_t* tokens_dev, int32_t* tokens_out);

/* Persistent multi-step decode: ONE resident launch runs up to n_steps greedy steps, each step's
 * token fed to the next step's embedding on the device, and ends early at a step boundary when
 * the host asks it to (the "Inference MegaKernel" page, section "MPK compiler and runtime": its
 * runtime's online mode keeps the kernel resident while tokens are pending and polls a host
 * shutdown signal instead of returning after every token).  Between steps every CTA waits for
 * all CTAs to retire the previous step (a grid-wide step word, release/acquire ordered); the
 * previous step's greedy token, the stop decision and the KV rows it appended are read after it.
 *
 * mk_decode_persistent_start enqueues the launch on the bound stream and returns at once.
 *  tokens, pos   HOST int32[batch]: the first step's tokens (in [0, vocab)) and positions
 *                (pos[b] + n_steps <= max_seq).  Step i decodes sequence b at pos[b] + i.
 *  n_steps       >= 1: the most steps the launch runs.
 *  logits        DEVICE fp32[batch, vocab], caller-owned: every step writes it; the last step's
 *                logits remain.
 *  tokens_dev    DEVICE int32[n_steps * batch], caller-owned, 4-byte aligned: step i's greedy
 *                tokens at [i * batch, (i + 1) * batch).  Must stay allocated until the wait.
 * While the launch is in flight the context accepts only mk_decode_persistent_stop,
 * mk_decode_persistent_progress and mk_decode_persistent_wait (other calls: MK_ERR_ARG).
 * Errors: MK_ERR_ARG (null or misaligned pointer, n_steps < 1, a token or position out of range,
 * a launch already in flight: nothing is launched), MK_ERR_POISONED, MK_ERR_CUDA. */
mk_status mk_decode_persistent_start(mk_ctx* c, const int32_t* tokens, const int32_t* pos, int32_t n_steps,
                                     float* logits, int32_t* tokens_dev);

/* Asks the in-flight launch to stop: the first step whose greedy token is chosen after the
 * request is the last one the launch runs (one or more steps always run).  A plain store to a
 * host word the device reads; returns at once.  MK_ERR_ARG if no launch is in flight. */
mk_status mk_decode_persistent_stop(mk_ctx* c);

/* Steps the in-flight (or last) launch has finished so far, read from a host word the device
 * writes after every step; does not wait.  MK_ERR_ARG on a null argument. */
mk_status mk_decode_persistent_progress(mk_ctx* c, int32_t* steps_done);

/* Waits for the launch to end.  steps_done (HOST int32, optional) receives the steps it ran
 * (1..n_steps); tokens_out (HOST int32[n_steps * batch], optional) their greedy tokens, step i at
 * [i * batch].  The context's next step continues the epoch after the last step run.  Errors:
 * MK_ERR_ARG (no launch in flight); a device error is reported as by mk_decode_step and poisons
 * the context. */
mk_status mk_decode_persistent_wait(mk_ctx* c, int32_t* steps_done, int32_t* tokens_out);

/* Asynchronous form: enqueues one step on the bound stream and returns.  next_tokens_dev is a
 * DEVICE int32[batch] buffer or NULL.  Device-side errors surface at the next mk_ctx_status or
 * mk_decode_step. */
mk_status mk_launch_step(mk_ctx* c, const int32_t* tokens, const int32_t* pos, float* logits,
                         int32_t* next_tokens_dev);

/* Waits for the bound stream and returns the device error state (MK_OK when no step failed).
 * info (optional, 8 int32): code, CTA, queue slot, counter, value seen, value wanted, role, 0.
 * role: 1 loader, 2 consumer (page / slot / CTA barrier), 3 publisher, 4 counter wait,
 * 5 tagged-data poll (counter, seen, wanted: -1, tag seen, tag wanted). */
mk_status mk_ctx_status(mk_ctx* c, int32_t* info);

/* Number of SMs of the current CUDA device (the natural sm_count), or MK_ERR_CUDA. */
mk_status mk_device_sm_count(int32_t* out);

/* The message of the calling thread's last non-OK status (thread-local; empty if none).  A
 * library convention with no counterpart on the page. */
const char* mk_last_error(void);

/* Ends a binding: asks a persistent launch in flight to stop, waits for the bound stream, then
 * frees the context's own device copies (queues, counter totals, layer table, step word) and its
 * pinned readback and control buffers.  The caller's weights, KV cache,
 * counters and scratch are not touched (the page's objects live as long as the request that bound
 * them; section "Hand-written whole-model MegaKernel", object table).  NULL is ignored. */
void mk_unbind(mk_ctx* c);

#ifdef __cplusplus
}
#endif
#endif /* MK_H */
