// Declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// Longest a pipeline wait may spin before the kernel gives up (flags
// PA_DEV_WAIT_TIMEOUT and skips the rest of its work).
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

constexpr int kMaxCtasPerSm = 8;
constexpr int kDefaultCtasPerSmMma = 4;  // default CTAs per SM on the bf16 tensor-core path
// Decode workspace: the status head, one merge counter per CTA, then two
// partial slots per CTA of the launch's grid (pa_decode_workspace_bytes sizes
// it for kMaxCtasPerSm CTAs on every SM, the largest grid); a slot is [G][D]
// floats of o plus [G][2] floats of (m, l).
constexpr int kSlotExtraFloatsPerHead = 2;
// floats of one partial slot, a multiple of 4 so that every slot is 16-byte aligned
inline __host__ __device__ size_t partial_slot_floats(int G, int D) {
    return ((size_t)G * (D + kSlotExtraFloatsPerHead) + 3) & ~(size_t)3;
}
constexpr int kMaxSmem = 227 * 1024;

// Cost weights of the range balance (see DecodeParams): 4 units a tile, and a
// segment's fixed work in units per compute path.  Measured per-CTA loop ends
// put a piece's fixed work near one tile of the stream on the tensor-core path
// (4 CTAs per SM) and near half a tile on the CUDA-core path (8 CTAs per SM).
// Over FP8 pools, where the consumer's instructions are the bound, a segment
// (its query rows, the softmax's end, the partial store and merge count) costs
// about six FP8 tiles: a fit of loop ends against tiles and segments per CTA
// gave 5.8, and a sweep of the weight was fastest at 24 units on all three
// unpartitioned workloads.
constexpr int kTileUnits = 4;
#ifndef PA_SEG_UNITS_MMA
#define PA_SEG_UNITS_MMA 4
#endif
#ifndef PA_SEG_UNITS_FMA
#define PA_SEG_UNITS_FMA 2
#endif
#ifndef PA_SEG_UNITS_FP8
#define PA_SEG_UNITS_FP8 24
#endif
constexpr int kMaxSegUnits = 4096;  // bound of pa_debug_set_seg_units
// Shares of the decode's CTAs by dispatch wave (the CTAs of a launch take the SMs in waves of one
// per SM): wave v of NWV takes kWaveWeight + skew (NWV - 1 - 2 v) parts.  An SM's warp scheduler
// favours the CTAs dispatched to it first, which on the issue-bound FP8 path end their equal
// shares several microseconds before the last-dispatched ones; the skew hands the first waves more.
// Measured over FP8 pools: skew 2 about 1.5 % faster on mha_b256_append, neutral elsewhere.
constexpr int kWaveWeight = 64;
#ifndef PA_WAVE_SKEW_FP8
#define PA_WAVE_SKEW_FP8 2
#endif

struct DecodeParams {
    void* out;
    const void* q;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    int32_t* status;    // workspace word 0
    // [num_ctas]: pieces of the split segment whose first piece CTA c holds that have been
    // stored so far; zero between calls (the CTA that completes the count resets it)
    int32_t* merge_counts;
    float* partials;    // [2 * num_ctas][G * (D + 2)]
    int32_t max_blocks_per_seq;
    int32_t max_len;  // min(max_seq_len, max_blocks_per_seq * block_size)
    int32_t num_seqs;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t num_blocks;
    int32_t group;            // G = num_q_heads / num_kv_heads
    int32_t partition_tiles;  // 0: split anywhere; else splits only at multiples of this
    int32_t num_ctas;
    // Without partitions, CTA ranges balance a cost in which a tile weighs
    // kTileUnits and every (sequence, KV head) segment seg_units more: the
    // fixed work of a piece (query load, softmax state, output store).
    int32_t seg_units;
    // ... and CTA c takes a share by its dispatch wave c / wave_ctas (see kWaveWeight)
    int32_t wave_ctas;
    int32_t wave_skew;
    float scale_log2;  // scale * log2(e) (times the K scale of an FP8 pool): scores in the base-2 domain
    float out_scale;   // multiplies the output: the V scale of an FP8 pool, else 1
    // time limit of the consumer's waits for query rows and tiles (the producer's
    // waits, and its final wait for the copies it issued, keep the full limit)
    uint64_t wait_limit_ns;
    // 1: split segments are merged inside the decode kernel (merge_counts); 0: by
    // merge_kernel, launched after it (the host picks per launch, see pa_api.cu)
    int32_t merge_in_kernel;
    // a host-built plan of this launch in device memory (pa_plan.h), or null: the kernels then
    // scan the lengths and search the CTA ranges themselves
    const int32_t* plan;
};

// One compiled decode kernel (dtype, head_dim, block_size, compute path).
// The merge of split segments when it is not done in the decode kernel: a
// second, small kernel (see pa_decode.cuh).
constexpr int kMergeThreads = 128;
// its shared memory for num_seqs sequences: the plan's prefix sums, the
// clamped lengths and the scan's warp sums
inline int merge_smem_bytes(int num_seqs, bool fixed) { return ((num_seqs + 1) * (fixed ? 2 : 1) + num_seqs + 8) * 4; }

// One compiled build of the decode kernel: its threads per CTA, ring stages and shared memory.
struct DecodeBuild {
    const void* kernel;
    int stages;
    int threads;
    int (*smem_bytes)(int num_seqs, bool fixed);
};

struct DecodeVariant {
    DecodeBuild in;            // merges split segments in the kernel (when merge_in_kernel_ok)
    DecodeBuild mk;            // launched when merge_kernel merges (may be the same kernel as `in`)
    const void* merge_kernel;  // launched right after the decode as its programmatic dependent, when used
    bool merge_in_kernel_ok;   // `in` has the in-kernel merge
    void (*launch)(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid, int smem,
                   int merge_grid, int merge_smem, cudaStream_t stream);
};

// Compiled variants.  `group` is Hq / Hkv; the CUDA-core path has exact
// instantiations for some group sizes and a run-time-group fallback.
bool decode_variant_f32(int head_dim, int block_size, int group, DecodeVariant* out);
bool decode_variant_f32_pow2(int head_dim, int block_size, int group, DecodeVariant* out);
bool decode_variant_bf16_mma(int head_dim, int block_size, DecodeVariant* out);
bool decode_variant_bf16_fma(int head_dim, int block_size, int group, DecodeVariant* out);
// bf16 queries and outputs over FP8 (E4M3) pools, CUDA-core path.
bool decode_variant_fp8(int head_dim, int block_size, int group, DecodeVariant* out);

// The decode of pa_decode_attention / _fp8 (pa_api.cu): checks, plan and launch.
// Refuses a workspace smaller than the bytes its own grid touches (the status
// head, a merge counter and two partial slots per CTA).  clear_status zeroes
// the status head and the merge counters on the stream after every check has
// passed, right before the launch.
constexpr size_t kStatusHeadBytes = 256;
pa_status decode_common(void* out, const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
                        int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t max_seq_len, int32_t num_seqs,
                        int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                        int32_t num_blocks, float scale, int32_t partition_tokens, void* workspace,
                        size_t workspace_bytes, pa_dtype dtype, float k_scale, float v_scale, void* stream,
                        bool clear_status, const void* plan = nullptr, size_t plan_bytes = 0);

// Host launch helpers shared by the attention entry points (pa_api.cu).
// The TMA map of a pool viewed as [num_blocks * Hkv * block_size][head_dim]
// rows, one box = block_size rows x 128 bytes with the 128-byte swizzle;
// cached per (device, pool, shape).
bool pool_map(CUtensorMap* map, int dev, const void* pool, int64_t rows, int head_dim, int block_size, pa_dtype dt);
// The TMA map of prefill query rows: q [tokens][heads][head_dim] bf16 viewed as
// (head_dim, heads, tokens), one box = 64 elements x box_heads x box_tokens with
// the 128-byte swizzle; cached per (device, q, shape).
bool prefill_q_map(CUtensorMap* map, int dev, const void* q, int64_t tokens, int heads, int head_dim, int box_heads,
                   int box_tokens);
// Opts the kernel into `smem` bytes of dynamic shared memory and returns its
// CTAs per SM; cached per (device, kernel, smem).
bool kernel_occupancy(int dev, const void* kernel, int threads, int smem, int* occ);

// Paged prefill (chunked causal) attention, bf16.
struct PrefillParams {
    void* out;
    const void* q;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const int32_t* cu_q_lens;
    int32_t* status;
    int32_t max_blocks_per_seq;
    int32_t num_seqs;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t num_blocks;
    int32_t group;          // G = num_q_heads / num_kv_heads
    int32_t tile_tokens;    // chunk tokens per 128-row query tile: 128 / G (rounded down)
    int32_t num_q_tokens;   // rows of q and out
    int32_t max_q_len;      // bound on every chunk (the grid is sized by it)
    int32_t out_align32;    // out is 32-byte aligned: 32-byte stores
    float scale_log2;
};

}  // namespace pa
