/*
 * pa.h -- C ABI of the paged KV-cache library (single GB300, sm_103a).
 *
 * The library implements the data-parallel hot path of PagedAttention as the
 * three PagedAttention pages describe it:
 *   [P1] "Q32: vLLM PagedAttention 原理" (agentalpha.top/interview/basics-tk516)
 *   [P2] "vLLM" (data.6616ai.com/article/vllm)
 *   [P3] "batch-008-day-02-interview-1" (ohmygp.com/posts/...)
 * Section names below refer to those pages.
 *
 * Conventions shared by every entry point
 *   - Device pointers are plain CUDA device addresses owned by the caller.
 *     The library never allocates, frees or retains device memory; each
 *     call only reads and writes the buffers it is given.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Device work is enqueued asynchronously on it; a PA_OK return
 *     means "validated and launched", not "finished".
 *   - Arguments are checked on the host before any launch; a failed check
 *     returns an error status and launches nothing.  A failed launch returns
 *     PA_ERR_CUDA.  No C++ exception crosses this interface.
 *   - Faults the host cannot see (a block id or slot outside the pool, a
 *     sequence length beyond its block table) are caught by bounds checks in
 *     the kernels: the offending access is skipped or clamped to block 0, and
 *     a bit is OR-ed into a caller-supplied int32 device status word
 *     (PA_DEV_* below).  The kernels never trap.
 *   - Layouts are contiguous row-major:
 *       K pool, V pool   [num_blocks][num_kv_heads][block_size][head_dim]
 *       q, out           [num_seqs][num_q_heads][head_dim]
 *       k_new, v_new     [num_tokens][num_kv_heads][head_dim]
 *       block_tables     int32 [num_seqs][max_blocks_per_seq]
 *       seq_lens         int32 [num_seqs]
 *       slot_mapping     int64 [num_tokens]
 *       src_dst_pairs    int32 [num_pairs][2]
 *     Device buffers must be 16-byte aligned.
 *   - Supported shapes for the device kernels: block_size 16 or 32,
 *     head_dim 64 or 128, num_q_heads a multiple of num_kv_heads with at most
 *     8 query heads per KV head; element type fp32 or bf16.  Anything else
 *     returns PA_ERR_UNSUPPORTED.
 *   - The host allocator is not thread-safe; callers serialise access to one
 *     allocator object.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_ABI_VERSION 1

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,        /* null pointer, negative size, misaligned buffer, ... */
    PA_ERR_UNSUPPORTED = 2,        /* shape or dtype outside the supported set */
    PA_ERR_OUT_OF_BLOCKS = 3,      /* the pool has too few free blocks (state unchanged) */
    PA_ERR_NO_SUCH_SEQ = 4,        /* unknown sequence id */
    PA_ERR_SEQ_EXISTS = 5,         /* sequence id already in use */
    PA_ERR_REFCOUNT_LIMIT = 6,     /* fork would push a block past the refcount cap */
    PA_ERR_WORKSPACE_TOO_SMALL = 7,/* decode workspace smaller than the launch needs (see pa_decode_workspace_bytes) */
    PA_ERR_BUFFER_TOO_SMALL = 8,   /* a host output array is too short */
    PA_ERR_CUDA = 9,               /* a CUDA runtime call or launch failed */
    PA_ERR_INTERNAL = 10,          /* unexpected host failure (e.g. host memory exhausted) */
    PA_ERR_SEQ_SWAPPED = 11        /* the sequence's blocks are swapped out (pa_seq_swap_out) */
} pa_status;

/* Element types.  PA_FP8_E4M3 (OCP FP8 E4M3 codes, one byte) is a pool type
 * only: pools of that type pair with bf16 queries and outputs through the
 * *_fp8 entry points. */
typedef enum pa_dtype { PA_F32 = 0, PA_BF16 = 1, PA_FP8_E4M3 = 2 } pa_dtype;

/* Bits of the device status word. */
#define PA_DEV_BAD_BLOCK_ID 0x1 /* a block id outside [0, num_blocks) was read or given */
#define PA_DEV_BAD_SLOT 0x2     /* a slot outside the pool was given */
#define PA_DEV_BAD_SEQ_LEN 0x4  /* seq_lens[b] < 0, or beyond its block table or max_seq_len */
#define PA_DEV_WAIT_TIMEOUT 0x8 /* an on-chip pipeline wait gave up (the output is not valid) */

/* ------------------------------------------------------------------------ */
/* Device kernels                                                            */
/* ------------------------------------------------------------------------ */

/*
 * Slot-mapped append ("reshape_and_cache").
 * [P3] 破局思路/按需分配: each decoded token takes one slot of the current
 * block; [P1] §2 非连续存储: new tokens are written into the block, existing
 * KV never moves.  For every token i with s = slot_mapping[i] >= 0:
 *     k_pool[s / block_size][h][s % block_size][:] = k_new[i][h][:]   for all h
 * and the same for V.  Negative slots are skipped (padding).  Bit-exact copy.
 * A slot >= num_blocks * block_size sets PA_DEV_BAD_SLOT and is skipped.
 * dev_status may be NULL (then out-of-range slots are skipped silently).
 * Slots of one call must be distinct (two tokens writing one slot race).
 */
pa_status pa_reshape_and_cache(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                               const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size, int32_t num_blocks, pa_dtype dtype,
                               int32_t* dev_status, void* stream);

/*
 * Copy-on-write block copy.
 * [P1] §3 Copy-on-Write, [P2] Copy-on-write 共享, [P3] 写时共享: a block shared
 * by several sequences is copied to a new physical block when one of them
 * writes into it.  For each pair p: pool[dst_p] = pool[src_p] over the whole
 * block (every KV head, all block_size slots, all of head_dim), K and V.
 * Bit-exact.  A block id outside [0, num_blocks) sets PA_DEV_BAD_BLOCK_ID and
 * that pair is skipped.  Destinations must be distinct and no destination
 * may be a source of the same call (the pairs are copied concurrently).
 * Enqueue it before the pa_reshape_and_cache that writes the same step's
 * tokens: a copy source may be written in place by its last sharer.
 */
pa_status pa_copy_blocks(void* k_pool, void* v_pool, const int32_t* src_dst_pairs, int32_t num_pairs,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                         pa_dtype dtype, int32_t* dev_status, void* stream);

/*
 * Size in bytes of the device workspace pa_decode_attention needs for these
 * shapes on the current CUDA device.  The workspace holds the status word
 * (first int32, in a 256-byte head), one merge counter (int32) per CTA of the
 * decode grid and two split-sequence partial slots per CTA; this size covers
 * the largest grid the device can take (8 CTAs on every SM), so it suffices
 * for every call with these head shapes whatever pa_decode_set_ctas_per_sm
 * says.  A call refuses (with PA_ERR_WORKSPACE_TOO_SMALL, before launching)
 * only a workspace smaller than what its own grid touches.  The caller
 * allocates it ONCE, zero-filled (the status word and the merge counters must
 * start at zero), and may reuse it across calls on one stream: the partial
 * slots are written before they are read, the status word only gathers error
 * bits, and every call leaves the merge counters at zero again (also when a
 * wait timed out: every piece is still stored and counted).
 */
pa_status pa_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                    int32_t head_dim, size_t* bytes_out);

/*
 * Paged decode attention, one query token per sequence.
 * [P2] 把虚拟内存搬进 KV Cache: the attention kernel reads KV by block index,
 * logically contiguous and physically scattered; [P1] follow-up 3
 * (FlashAttention): KV is loaded block by block with the pointer indexing
 * adapted to non-contiguous blocks.  For each sequence b and query head h,
 * with g = h / (num_q_heads / num_kv_heads) and token t < seq_lens[b] in
 * physical block block_tables[b][t / block_size] at offset t % block_size:
 *     s_t = scale * q[b][h] . K[t],   out[b][h] = sum_t softmax(s)_t V[t]
 * computed with an online (running max and sum) softmax in fp32, inputs in
 * `dtype`, output in `dtype` (bf16 rounds to nearest even).  An empty
 * sequence gives a zero output.
 * Long sequences are split across CTAs (flash-decoding) and the partial
 * results merged on the device, in one of two ways chosen per call from the
 * shapes and the grid: in the decode kernel itself (each piece of a split
 * (sequence, KV head) segment is stored to the workspace and counted on the
 * segment's counter; the CTA whose piece completes the count combines the
 * pieces and writes the segment's output rows), or by a second kernel
 * launched right after the decode kernel as its programmatic dependent, which
 * waits for the decode grid to finish and writes the output rows of split
 * segments.  partition_tokens = 0 splits anywhere on a
 * block boundary, so that every CTA gets the same share of blocks plus a
 * fixed cost per (sequence, KV head) it touches; partition_tokens = P > 0
 * (a multiple of block_size) allows splits only at multiples of P tokens.
 * max_seq_len bounds every seq_lens[b]; a larger or negative length sets
 * PA_DEV_BAD_SEQ_LEN and is clamped.  Table entries read for t < seq_len
 * must be in [0, num_blocks); others set PA_DEV_BAD_BLOCK_ID.
 * workspace: see pa_decode_workspace_bytes; its first int32 is the status
 * word.  Concurrent calls must use different workspaces.
 * The kernel is launched as a programmatic dependent of the preceding kernel
 * on `stream`: when that kernel allows an early start (pa_reshape_and_cache
 * does), this one computes its work split from seq_lens and block_tables and
 * starts reading them while that kernel finishes; it reads the pools and q,
 * and writes out and the workspace, only after that kernel has completed.  So
 * a kernel that allows early start must not write seq_lens or block_tables.
 */
pa_status pa_decode_attention(void* out, const void* q, const void* k_pool, const void* v_pool,
                              const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                              int32_t max_seq_len, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
                              int32_t partition_tokens, void* workspace, size_t workspace_bytes, pa_dtype dtype,
                              void* stream);

/*
 * A host-built work plan for one pa_decode_attention (or _fp8) call, and
 * the calls that take it.  A decode launch first scans seq_lens into
 * per-sequence block prefix sums, searches each CTA's range of the tile
 * list, walks to its first piece and fetches that piece's block-table
 * entries: four dependent steps before the first tile is requested.  The
 * host allocator already holds every length and table entry (it exported
 * them), so it can compute all of that; the launch then reads it in one
 * round trip.  (The pages have no counterpart: an optimisation of the
 * decode's start, not a change to what it computes.)
 *
 * pa_decode_plan_bytes: the plan's size for these shapes on the current
 * device (it holds one 160-byte record per CTA of the launch's grid).
 *
 * pa_decode_build_plan: writes the plan into plan_out (host memory, 4-byte
 * aligned, plan_bytes long) from HOST copies of block_tables
 * ([num_seqs][max_blocks_per_seq]) and seq_lens, equal to the device copies
 * the call will read.  max_seq_len, partition_tokens and dtype (the pool's:
 * PA_F32, PA_BF16 or PA_FP8_E4M3) must be the call's.  Returns
 * PA_ERR_WORKSPACE_TOO_SMALL if plan_bytes is short; out-of-range lengths are
 * clamped as the decode clamps them (the decode still flags them).
 *
 * pa_decode_attention_planned / pa_decode_attention_fp8_planned: the decode
 * calls with a device copy of that plan (4-byte aligned, plan_bytes long;
 * shorter is PA_ERR_INVALID_ARG).  A plan whose header does not name this
 * call's batch size, grid, KV heads, partition size, segment weight, block
 * size, length bound, table width, merge mode, wave size and wave skew is
 * ignored (the launch computes its own);
 * a plan built from other lengths or table entries than the device copies
 * hold gives wrong outputs: rebuild it whenever either changes.  The launch
 * trusts a matching plan's prefix sums (only its block ids are checked, as
 * table entries are), so a buffer not written by pa_decode_build_plan for
 * these inputs may make it read block_tables out of range.  Everything
 * else is as for pa_decode_attention and pa_decode_attention_fp8; the results
 * are bit for bit those of the unplanned calls.
 */
pa_status pa_decode_plan_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t block_size, int32_t max_blocks_per_seq, int32_t max_seq_len,
                               int32_t partition_tokens, pa_dtype dtype, size_t* bytes_out);
pa_status pa_decode_build_plan(const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                               int32_t max_seq_len, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size, int32_t partition_tokens, pa_dtype dtype,
                               void* plan_out, size_t plan_bytes);
pa_status pa_decode_attention_planned(void* out, const void* q, const void* k_pool, const void* v_pool,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* seq_lens, int32_t max_seq_len, int32_t num_seqs,
                                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, int32_t num_blocks, float scale, int32_t partition_tokens,
                                      void* workspace, size_t workspace_bytes, pa_dtype dtype, const void* plan,
                                      size_t plan_bytes, void* stream);
pa_status pa_decode_attention_fp8_planned(void* out, const void* q, const void* k_pool, const void* v_pool,
                                          float k_scale, float v_scale, const int32_t* block_tables,
                                          int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t max_seq_len,
                                          int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
                                          int32_t partition_tokens, void* workspace, size_t workspace_bytes,
                                          const void* plan, size_t plan_bytes, void* stream);

/*
 * Paged decode attention without a caller-supplied workspace.  The pages have
 * no counterpart to this entry point: it exists for callers that cannot
 * allocate device memory, such as a plugin inside a framework that owns every
 * device allocation, or a serving loop that must not allocate once running.
 * Arguments and results are those of pa_decode_attention, minus the
 * workspace.  Its scratch is a static buffer of PA_STATIC_WORKSPACE_BYTES
 * (8 MiB) in the library's device image, held on every GPU that loads the
 * library until the process exits.  A call whose decode grid needs more
 * scratch than that (the status head, then per CTA a merge counter and two
 * partial slots of G * (head_dim + 2) floats) returns
 * PA_ERR_WORKSPACE_TOO_SMALL before anything runs; on a 152-SM GB300 every
 * supported shape fits at the default CTAs per SM.  The call allocates
 * nothing: after its argument checks it clears the status head and the merge
 * counters of the buffer (one cudaMemsetAsync) and enqueues the decode.
 * That memset sits between the decode and the kernel before it on the
 * stream, so unlike pa_decode_attention this call does not overlap its start
 * with a preceding pa_reshape_and_cache.  If
 * dev_status_out is not NULL, the call's device status word (PA_DEV_* bits)
 * is copied there on `stream` afterwards.
 * The first call on a device looks up the buffer's device address; make that
 * first call before any stream capture.  Every call on a device shares the
 * one buffer, so calls that can overlap on the GPU (different streams, or
 * concurrent host threads) race: serialise them.
 */
#define PA_STATIC_WORKSPACE_BYTES (8u << 20)
pa_status pa_decode_attention_static(void* out, const void* q, const void* k_pool, const void* v_pool,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                     int32_t max_seq_len, int32_t num_seqs, int32_t num_q_heads,
                                     int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                     float scale, int32_t partition_tokens, pa_dtype dtype, int32_t* dev_status_out,
                                     void* stream);

/*
 * Launch facts of pa_decode_attention for these shapes on the current device
 * (no launch): CTAs in the grid, pipeline stages per CTA (on the tensor-core
 * path at block size 16 a stage holds two blocks' tiles), dynamic shared
 * memory per CTA in bytes, and 1 if the tensor-core (mma) path is used, else
 * 0 (CUDA-core FMA path).  max_blocks_per_seq bounds the blocks of every
 * sequence; partition_tokens is as for pa_decode_attention (the build and the
 * grid can depend on it).  Any output pointer may be NULL.
 */
pa_status pa_decode_launch_info(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                int32_t block_size, int32_t max_blocks_per_seq, int32_t partition_tokens,
                                pa_dtype dtype, int32_t* ctas, int32_t* stages, int32_t* smem_bytes,
                                int32_t* uses_mma);

/*
 * Kernels one pa_decode_attention (or _fp8, _static) call with these shapes
 * launches on the current device (no launch): 1 when it merges split
 * segments in the decode kernel, 2 when the merge kernel follows it.
 * max_blocks_per_seq bounds the blocks of every sequence, as for
 * pa_decode_launch_info.  partition_tokens: as for pa_decode_attention.
 */
pa_status pa_decode_kernels_per_call(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                     int32_t block_size, int32_t max_blocks_per_seq, int32_t partition_tokens,
                                     pa_dtype dtype, int32_t* kernels);

/*
 * Tuning: CTAs per SM of the decode grid (1..8; 0 restores the default: 4 on
 * the bf16 tensor-core path, otherwise, FP8 pools included, as many as fit,
 * at most 8).  Process-wide; affects later pa_decode_attention and
 * pa_decode_attention_fp8 calls.  More CTAs per SM keep more tiles in flight
 * but add split points (partials) at CTA edges.
 */
pa_status pa_decode_set_ctas_per_sm(int32_t ctas);

/*
 * Testing aid for failure detection (no counterpart on the pages): the time
 * limit, in nanoseconds, of the decode kernel's waits for its query rows and
 * KV tiles (consumer side).  Every on-chip wait of the kernels is bounded; one
 * that runs out sets PA_DEV_WAIT_TIMEOUT in the status word, the CTA stops
 * issuing and consuming, waits (with the full limit) for the copies it has
 * already issued, and exits, so the context stays usable and the output of
 * that call is not valid.  A limit far below a DRAM round trip makes the waits
 * run out on purpose.  0 restores the default (2 s); values above it return
 * PA_ERR_INVALID_ARG.  Process-wide; affects later pa_decode_attention,
 * pa_decode_attention_fp8 and pa_decode_attention_static calls.
 */
pa_status pa_debug_set_wait_limit_ns(uint64_t ns);

/*
 * Testing aid (no counterpart on the pages): where pa_decode_attention,
 * pa_decode_attention_fp8 and pa_decode_attention_static merge split
 * segments.  0: chosen per call (the default); 1: always in the decode
 * kernel; 2: always by the second kernel.  Results agree within rounding
 * order.  Other values return PA_ERR_INVALID_ARG.  Process-wide.
 */
pa_status pa_debug_set_merge_mode(int32_t mode);

/*
 * Tuning aid (no counterpart on the pages): the weight of one (sequence, KV
 * head) segment in the balance of the decode's CTA ranges, in units of which
 * a tile weighs 4.  0 restores each compute path's own weight; 1 .. 4096 sets
 * it for every later pa_decode_attention, pa_decode_attention_fp8,
 * pa_decode_attention_static and pa_decode_build_plan call (a plan records
 * the weight it was built with and is used only by calls with the same one).
 * Results agree within rounding order.  Other values return
 * PA_ERR_INVALID_ARG.  Process-wide.
 */
pa_status pa_debug_set_seg_units(int32_t units);

/*
 * Tuning aid (no counterpart on the pages): the skew of the decode's CTA
 * shares by dispatch wave.  A launch's CTAs take the SMs in waves of one per
 * SM, and an SM's warp scheduler favours the CTAs dispatched to it first;
 * without partitions, wave v of n then takes 64 + skew (n - 1 - 2 v) parts of
 * the work (equal parts at skew 0; the shares stay equal whenever the lightest
 * range would be under one tile).  -1 restores each compute path's own skew;
 * 0 .. 8 sets it for every later decode call and pa_decode_build_plan (a plan
 * records the skew and the wave size it was built with and is used only by
 * calls with the same).  Results agree within rounding order.  Other values
 * return PA_ERR_INVALID_ARG.  Process-wide.
 */
pa_status pa_debug_set_wave_skew(int32_t skew);

/*
 * Testing aid (no GPU needed): the decode's CTA ranges as a launch computes
 * them, from block_counts[num_seqs] (blocks per sequence, per KV head) and the
 * launch's grid (num_ctas), segment weight, partition size (in tiles, 0 for
 * none), wave size and skew.  Writes the working CTAs' count to
 * *working_ctas_out (W <= num_ctas), their range starts to starts_out[0 .. W]
 * (tile indices; starts_out needs num_ctas + 1 entries), and, when owners_out
 * is not null, the owning CTA of every tile (owners_cap entries at least;
 * PA_ERR_WORKSPACE_TOO_SMALL otherwise).  Tiles are numbered sequence-major,
 * then KV head, then block.  Bad arguments return PA_ERR_INVALID_ARG.
 */
pa_status pa_debug_plan_ranges(const int32_t* block_counts, int32_t num_seqs, int32_t num_kv_heads,
                               int32_t partition_tiles, int32_t seg_units, int32_t num_ctas, int32_t wave_ctas,
                               int32_t wave_skew, int64_t* starts_out, int32_t* owners_out, size_t owners_cap,
                               int32_t* working_ctas_out);

/*
 * FP8 KV pools (an extrapolation: the pages list FP8 among the quantisation
 * formats the ecosystem supports, data.6616ai.com "PagedAttention 之外").
 * Pools hold OCP E4M3 codes (PA_FP8_E4M3, one byte per element, head_dim
 * 128), one fp32 scale per pool: element x is stored as the code of
 * fp32(x / scale), rounded to nearest (ties to even) and saturated to +-448,
 * and read back as value(code) * scale.
 *
 * pa_reshape_and_cache_fp8: the slot-mapped append of pa_reshape_and_cache
 * with that quantisation; k_new / v_new are in_dtype (bf16 or fp32)
 * [N][Hkv][128].  The codes are bit-exact against the definition.
 *
 * pa_decode_attention_fp8: pa_decode_attention over FP8 pools with bf16 q
 * and out: out = softmax(scale q . (K code values * k_scale)) (V code values
 * * v_scale).  Same layouts, workspace (pa_decode_workspace_bytes), split
 * modes and error reporting.  Every group size runs on the tensor cores:
 * the codes are widened to f16 in registers and the MMAs run in f16 (the
 * bf16 queries are rounded to f16, so their magnitudes must stay within f16
 * range).  k_scale and v_scale must be finite and > 0.
 */
pa_status pa_reshape_and_cache_fp8(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                                   const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t block_size, int32_t num_blocks, pa_dtype in_dtype,
                                   float k_scale, float v_scale, int32_t* dev_status, void* stream);
pa_status pa_decode_attention_fp8(void* out, const void* q, const void* k_pool, const void* v_pool, float k_scale,
                                  float v_scale, const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* seq_lens, int32_t max_seq_len, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  int32_t num_blocks, float scale, int32_t partition_tokens, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * Swap a preempted sequence's blocks out to a block store and back
 * (data.6616ai.com "PagedAttention 之外": KV swapped to CPU memory under
 * memory pressure and restored to resume).
 *
 * pa_swap_out: for i < num, store[i] = pool[blocks[i]] over the whole block
 * (every KV head, all block_size slots, all of head_dim), K and V.  Any pool
 * dtype, FP8 included (pa_copy_blocks likewise).
 * pa_swap_in:  for i < num, pool[blocks[i]] = store[i].  Bit-exact.
 * The stores are [num][num_kv_heads][block_size][head_dim] in the pools'
 * dtype and may be pinned host memory (cudaHostAlloc / pinned tensors): the
 * kernels read or write it directly over the host link, with no device
 * staging.  blocks (int32 [num]) must be device-accessible (device memory or
 * pinned host memory).  Use the ids pa_seq_swap_out / pa_seq_swap_in return,
 * enqueued in that order on the stream.  A block id outside [0, num_blocks)
 * sets PA_DEV_BAD_BLOCK_ID in *dev_status (if not NULL) and that block is
 * skipped.  Blocks of one call must be distinct for pa_swap_in.  num <= 65535.
 */
pa_status pa_swap_out(const void* k_pool, const void* v_pool, const int32_t* blocks, int32_t num, void* k_store,
                      void* v_store, int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                      pa_dtype dtype, int32_t* dev_status, void* stream);
pa_status pa_swap_in(const void* k_store, const void* v_store, const int32_t* blocks, int32_t num, void* k_pool,
                     void* v_pool, int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
                     pa_dtype dtype, int32_t* dev_status, void* stream);

/*
 * Paged prefill (chunked causal) attention, bf16.
 *
 * "Q32: vLLM PagedAttention 原理" follow-up 3 (FlashAttention loads the KV
 * cache block by block, adapted to non-contiguous blocks) and
 * data.6616ai.com "把虚拟内存搬进 KV Cache" (attention reads KV by block
 * index).  Sequence b holds seq_lens[b] tokens in the pools, its K/V already
 * appended (pa_reshape_and_cache); the last n_b = cu_q_lens[b+1] - cu_q_lens[b]
 * of them are a chunk whose queries are given.  Chunk token i sits at position
 * p = seq_lens[b] - n_b + i and attends to the keys at positions 0..p:
 *     out[cu_q_lens[b] + i][h] = softmax_{t <= p}(scale q . K[t]) V[t],
 * with query head h reading KV head h / (num_q_heads / num_kv_heads).
 *
 * Layouts (device, row-major, caller-owned): q and out [T][num_q_heads][head_dim]
 * bf16 with T = cu_q_lens[num_seqs]; pools as for pa_decode_attention;
 * block_tables int32 [num_seqs][max_blocks_per_seq]; seq_lens int32 [num_seqs];
 * cu_q_lens int32 [num_seqs + 1], non-decreasing from 0; num_q_tokens = T,
 * the rows of q and out.  max_q_len bounds every n_b (the grid is sized by
 * it).  Supported: bf16, head_dim 64 or 128, block_size 16 or 32,
 * num_q_heads / num_kv_heads <= 8, num_seqs <= 65535.
 *
 * scale must be finite and > 0 (the kernel folds it into one fma per weight
 * against the raw row maximum); otherwise PA_ERR_INVALID_ARG.
 * Runs on the fifth-generation tensor cores (tcgen05.mma with TMEM
 * accumulators), one persistent CTA per SM.
 *
 * Errors: host checks return a status before any launch.  A sequence with
 * n_b > seq_lens[b], n_b > max_q_len, rows past num_q_tokens, or seq_lens[b]
 * beyond its block table sets PA_DEV_BAD_SEQ_LEN in *dev_status (if not NULL)
 * and its rows are not written; block ids outside [0, num_blocks) set PA_DEV_BAD_BLOCK_ID and block
 * 0 is read instead; a pipeline wait that gives up sets PA_DEV_WAIT_TIMEOUT.
 * Asynchronous on `stream` (cudaStream_t).  Allocates nothing.
 */
pa_status pa_prefill_attention(void* out, const void* q, const void* k_pool, const void* v_pool,
                               const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                               const int32_t* cu_q_lens, int32_t num_seqs, int32_t num_q_tokens, int32_t max_q_len,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int32_t num_blocks, float scale, pa_dtype dtype, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------ */
/* Host block allocator                                                      */
/* ------------------------------------------------------------------------ */
/*
 * [P1] §2 分块管理/Block Table映射, [P2] 把虚拟内存搬进 KV Cache, [P3] 按需分配/
 * 块表映射/写时共享.  Blocks are taken on demand, only when a sequence's tail
 * block is full; each sequence keeps a block table (logical -> physical);
 * forked sequences share blocks through reference counts, and a write into
 * a block with refcount > 1 first copies it (copy-on-write).
 * Readings of points the pages leave open:
 *   - The free list is a FIFO queue: allocation pops the front, a freed block
 *     is pushed at the back.  Its initial order is the caller's (free_order),
 *     or 0..num_blocks-1.
 *   - Append of one token to sequence s with length n: if n % block_size == 0
 *     a new block is pushed onto the table; otherwise, if the tail block's
 *     refcount is > 1, a new block d is taken, the pair (tail, d) is emitted,
 *     the tail's refcount drops by one and the table entry points at d.  The
 *     token's slot is table[n / block_size] * block_size + n % block_size.
 *     So the last remaining sharer writes in place and a full shared block
 *     is never copied.
 *   - Fork copies the parent's table and length, adding one reference to
 *     each block.  Free walks the table in logical order, dropping one
 *     reference per block; blocks reaching zero go to the back of the free
 *     list.
 *   - Every call is all-or-nothing: on any error the allocator is unchanged.
 * The allocator owns only host memory.
 */
typedef struct pa_allocator pa_allocator;

typedef struct pa_alloc_stats_t {
    int32_t num_blocks;
    int32_t block_size;
    int32_t free_blocks;   /* on the free list (cached evictable blocks are not) */
    int32_t used_blocks;   /* blocks with refcount > 0 */
    int32_t shared_blocks; /* blocks with refcount > 1 */
    int32_t num_seqs;
    int64_t tokens;        /* sum of the sequences' lengths (swapped-out ones included) */
    int64_t slots;         /* used_blocks * block_size */
    int64_t cow_copies;    /* copy-on-write pairs emitted since creation */
} pa_alloc_stats_t;

/* free_order: num_blocks distinct ids (a permutation of 0..num_blocks-1), or NULL. */
pa_status pa_alloc_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order, pa_allocator** out);
void pa_alloc_destroy(pa_allocator* a);
/* Optional cap on a block's refcount (0 = none); fork fails with PA_ERR_REFCOUNT_LIMIT past it. */
pa_status pa_alloc_set_max_refcount(pa_allocator* a, int32_t max_refcount);
pa_status pa_seq_create(pa_allocator* a, int64_t seq_id);
/*
 * Append n_tokens to one sequence.  slots_out receives n_tokens slots;
 * cow_pairs_out receives up to n_tokens (src, dst) pairs (at most one per
 * call is possible) and *n_cow_out their count.
 */
pa_status pa_seq_append(pa_allocator* a, int64_t seq_id, int32_t n_tokens, int64_t* slots_out,
                        int32_t* cow_pairs_out, int32_t* n_cow_out);
/* One token for each of n ids, processed in the given order; arrays as above, sized n. */
pa_status pa_append_batch(pa_allocator* a, const int64_t* seq_ids, int32_t n, int64_t* slots_out,
                          int32_t* cow_pairs_out, int32_t* n_cow_out);
pa_status pa_seq_fork(pa_allocator* a, int64_t parent, int64_t child);
pa_status pa_seq_free(pa_allocator* a, int64_t seq_id);
/* Copies the block table (cap entries at most) and its length into *n_out. */
pa_status pa_seq_block_table(const pa_allocator* a, int64_t seq_id, int32_t* out, int32_t cap, int32_t* n_out);
pa_status pa_seq_len(const pa_allocator* a, int64_t seq_id, int32_t* len_out);
/*
 * Block tables and lengths of n sequences in the layout pa_decode_attention
 * reads: tables_out [n][max_blocks_per_seq] (unused entries set to 0) and
 * lens_out [n].  PA_ERR_BUFFER_TOO_SMALL if a table is longer than
 * max_blocks_per_seq.
 */
pa_status pa_export_tables(const pa_allocator* a, const int64_t* seq_ids, int32_t n, int32_t max_blocks_per_seq,
                           int32_t* tables_out, int32_t* lens_out);
/*
 * Swap-out of a preempted sequence (data.6616ai.com "PagedAttention 之外":
 * when memory runs short the scheduler swaps a request's KV out to CPU memory
 * and swaps it back in to resume; "可能的追问": low-priority requests' KV is
 * moved to the CPU, then restored).
 *
 * pa_seq_swap_out writes the sequence's block table (physical ids in logical
 * order, *n_out of them, cap at most) to blocks_out and then drops the
 * sequence's references as pa_seq_free does (a block whose refcount reaches 0
 * returns to the back of the free list).  The sequence keeps its id and length
 * but holds no blocks: append, fork, block_table and export_tables on it
 * return PA_ERR_SEQ_SWAPPED until pa_seq_swap_in.  The caller copies those
 * blocks out (pa_swap_out) on the stream before anything that may reuse them.
 *
 * pa_seq_swap_in takes ceil(len / block_size) fresh blocks from the free list
 * (refcount 1 each, so a block that was shared before the swap-out comes back
 * private), makes them the sequence's table and writes them to blocks_out;
 * the caller copies the saved contents in (pa_swap_in).  PA_ERR_OUT_OF_BLOCKS
 * or PA_ERR_BUFFER_TOO_SMALL leave the state unchanged (*n_out still says how
 * many blocks are needed); PA_ERR_INVALID_ARG if the sequence is not swapped.
 */
pa_status pa_seq_swap_out(pa_allocator* a, int64_t seq_id, int32_t* blocks_out, int32_t cap, int32_t* n_out);
pa_status pa_seq_swap_in(pa_allocator* a, int64_t seq_id, int32_t* blocks_out, int32_t cap, int32_t* n_out);
/*
 * Prefix caching (data.6616ai.com, paging's second dividend: the KV blocks of
 * a prefix common to many requests, such as a system prompt, are cached and
 * reused across requests, so prefill computes only what is not cached).
 *
 * A full block is identified by the token ids of the whole prefix it
 * completes (a chained 64-bit hash, every hit verified against the stored
 * tokens and parent hash).  pa_seq_cache_prefix registers the first
 * n_tokens / block_size full blocks of a sequence whose first n_tokens KV
 * entries hold `tokens` (call it once they are written); a prefix already in
 * the cache keeps its entry.  pa_seq_create_cached creates a sequence whose
 * table starts with the longest run of cached blocks matching `tokens`, at
 * most (n_tokens - 1) / block_size of them so that at least one prompt token
 * is left to compute, each taking one more reference; *n_cached_out gets the
 * tokens covered (a multiple of block_size), which become the sequence's
 * length.  The caller appends the other n_tokens - *n_cached_out tokens and
 * prefills them as one chunk (pa_prefill_attention).
 *
 * A cached block whose last reference goes is not freed: it stays cached and
 * evictable.  An allocation takes the free list first, then evicts the cached
 * block released longest ago, which also leaves the cache.  Without
 * registered blocks the allocator behaves exactly as described above.
 * pa_prefix_cache_stats reports the cached and the evictable block counts
 * (either pointer may be NULL).
 */
pa_status pa_seq_create_cached(pa_allocator* a, int64_t seq_id, const int32_t* tokens, int32_t n_tokens,
                               int32_t* n_cached_out);
pa_status pa_seq_cache_prefix(pa_allocator* a, int64_t seq_id, const int32_t* tokens, int32_t n_tokens);
pa_status pa_prefix_cache_stats(const pa_allocator* a, int32_t* cached_blocks, int32_t* evictable_blocks);
/* Refcount of a block, or -1 if the id is out of range. */
int32_t pa_block_refcount(const pa_allocator* a, int32_t block);
pa_status pa_alloc_stats(const pa_allocator* a, pa_alloc_stats_t* out);
/* The free list in pop order (cap entries at most); count in *n_out. */
pa_status pa_alloc_free_list(const pa_allocator* a, int32_t* out, int32_t cap, int32_t* n_out);

/* ------------------------------------------------------------------------ */
const char* pa_status_str(pa_status s);
int32_t pa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
