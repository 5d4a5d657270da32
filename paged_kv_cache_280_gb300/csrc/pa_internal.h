// Declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

constexpr int kMaxCtasPerSm = 4;  // bound used to size the decode workspace
constexpr int kMaxSmem = 227 * 1024;

struct DecodeParams {
    void* out;
    const void* q;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    int32_t* status;    // workspace word 0
    int32_t* counters;  // [num_seqs * num_kv_heads], zero between calls
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
    float scale_log2;  // scale * log2(e): scores are kept in the base-2 domain
};

// One compiled decode kernel (dtype, head_dim, block_size, compute path).
struct DecodeVariant {
    const void* kernel;
    int stages;
    int threads;
    int (*smem_bytes)(int num_seqs, bool fixed);
    void (*launch)(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid, int smem,
                   cudaStream_t stream);
};

bool decode_variant_f32(int head_dim, int block_size, DecodeVariant* out);
bool decode_variant_bf16(int head_dim, int block_size, bool mma, DecodeVariant* out);

}  // namespace pa
