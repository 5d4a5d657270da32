// Paged prefill (chunked causal) attention for sm_103a, bf16, on the
// fifth-generation tensor cores.
//
// What it computes ("Q32: vLLM PagedAttention 原理" follow-up 3: FlashAttention
// loads the KV cache block by block, its block loading adapted to
// non-contiguous storage; data.6616ai.com "把虚拟内存搬进 KV Cache": attention
// reads KV by block index): sequence b holds seq_lens[b] tokens in the paged
// pool, the last n_b = cu_q_lens[b+1] - cu_q_lens[b] of them are a chunk
// whose queries are given, and chunk token i (position p = seq_lens[b] - n_b
// + i) attends to the keys at positions 0..p:  out = softmax(scale q K^T) V.
//
// Work decomposition.  For one (sequence, KV head) the G query heads of each
// chunk token are stacked into rows (token-major), and a CTA takes a tile of
// 128 rows (128 / G chunk tokens): the M of every MMA, one row per TMEM lane.
// All rows of a tile share each K/V stage, so S = Q K^T and O = P V are dense
// 128-row contractions.  Tiles that end later in the chunk see more keys; the
// grid hands them out first.  Two CTAs share an SM, so one's softmax overlaps
// the other's MMAs.
//
// CTA: six warps.
//   - Producer (warp 4): walks the block table and moves 64 keys of K and V per
//     stage with TMA (cp.async.bulk.tensor, 128-byte swizzle, evict-last L2
//     policy: the segment's other tiles read the same blocks) into a 2-stage
//     ring guarded by full / empty mbarriers.
//   - MMA (warp 5, one thread): S_j = Q K_j^T into one of two TMEM buffers
//     (M 128, N 64, K = head_dim), issued one stage ahead of the softmax; then
//     O += P_j V_j (M 128, N = head_dim, K 64) with P_j from shared memory and
//     V_j an MN-major operand.  Completion is signalled by tcgen05.commit.
//   - Softmax (warps 0-3, one thread per query row): loads the tile's Q rows
//     into the swizzled layout once; per stage reads its S row from TMEM,
//     applies the causal mask and scale, keeps a running max and sum in the
//     base-2 domain, and writes its row of P (bf16) over the stage's K, which
//     S_j has finished reading.  O is rescaled in TMEM only when a row's max
//     grows by more than 2^8 (the weights stay <= 256, exact in the final
//     ratio); the final O / l is written from TMEM.  On the stage that holds
//     the tile's last position it zeroes the V rows past it: their slots may
//     hold any bits, and zero weight times NaN is NaN.
// Every wait is bounded; a timeout sets PA_DEV_WAIT_TIMEOUT, every role stops,
// and the CTA waits for its own copies and MMAs before freeing TMEM.
#include <cmath>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kPfSoftmaxWarps = 4;
constexpr int kPfProducer = 4;  // warp index
constexpr int kPfMma = 5;       // warp index
constexpr int kPfThreads = 192;
constexpr int kPfRows = 128;    // query rows per CTA = MMA M = TMEM lanes
constexpr int kPfKeys = 64;     // keys per stage: N of S, K of P V
constexpr int kPfStages = 2;
constexpr int kPfCtasPerSm = 2;
constexpr uint32_t kPfTmemCols = 256;  // O in columns [0, D), S buffer i in [128 + 64 i, 192 + 64 i)
constexpr uint32_t kPfTmemS = 128;
constexpr float kPfRescaleLog2 = 8.f;  // rescale O only when a row max grows by more than this (log2)

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 2^x on the SFU (ex2.approx: a few ulp, well inside the bf16 output bound); 2^-inf = +0.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Shared memory of one CTA (1024-byte aligned regions, 128-byte swizzle):
//   Q      [D / 64 panels][128 rows][128 B]
//   stage  K|P: K as [D / 64 panels][64 keys][128 B], later P as [128 rows][128 B]
//          V:   [D / 64 panels][64 keys][128 B]
template <int D, int BS>
struct PfLayout {
    static constexpr int kPanels = D / 64;
    static constexpr int kQPanel = kPfRows * 128;
    static constexpr int kKVPanel = kPfKeys * 128;
    static constexpr int kQBytes = kPanels * kQPanel;
    static constexpr int kKBytes = kPanels * kKVPanel;
    static constexpr int kPBytes = kPfRows * kPfKeys * 2;
    static constexpr int kKPBytes = kKBytes > kPBytes ? kKBytes : kPBytes;
    static constexpr int kVBytes = kPanels * kKVPanel;
    static constexpr int kStageBytes = kKPBytes + kVBytes;
    static constexpr int kBlocksPerStage = kPfKeys / BS;
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = kQBytes;
    static constexpr int kBarOff = kRingOff + kPfStages * kStageBytes;
    // mbarriers: kv_full[2], kv_empty[2], s_full[2], s_free[2], p_ready[2], o_done, o_final, q_ready, mma_drain
    static constexpr int kNumBars = 5 * kPfStages + 4;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // abort flag, TMEM address
    static constexpr int kUsed = kMiscOff + 64 + 1024;       // +1 KB to align the base
    // at least a third of the SM's shared memory, so that no third CTA (and no TMEM request
    // beyond the SM's 512 columns) lands on an SM
    static constexpr int kBytes = kUsed > 80 * 1024 ? kUsed : 80 * 1024;
    static_assert(kQPanel % 1024 == 0 && kKVPanel % 1024 == 0 && kStageBytes % 1024 == 0, "1024-byte alignment");
};

struct PfBars {
    uint32_t base;
    __device__ uint32_t kv_full(int s) const { return base + 8u * s; }
    __device__ uint32_t kv_empty(int s) const { return base + 8u * (kPfStages + s); }
    __device__ uint32_t s_full(int s) const { return base + 8u * (2 * kPfStages + s); }
    __device__ uint32_t s_free(int s) const { return base + 8u * (3 * kPfStages + s); }
    __device__ uint32_t p_ready(int s) const { return base + 8u * (4 * kPfStages + s); }
    // phase k completes with P_k V_k
    __device__ uint32_t o_done() const { return base + 8u * (5 * kPfStages); }
    // its one phase completes with the last P V
    __device__ uint32_t o_final() const { return base + 8u * (5 * kPfStages + 1); }
    __device__ uint32_t q_ready() const { return base + 8u * (5 * kPfStages + 2); }
    __device__ uint32_t mma_drain() const { return base + 8u * (5 * kPfStages + 3); }
};

// Warp-collective bounded wait (every lane calls it); gives up once the CTA's abort flag is set.
__device__ __forceinline__ bool pf_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag, int32_t* status) {
    if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
    bool ok = mbar_wait(bar, parity, kWaitLimitNs, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
        *abort_flag = 1;
        if ((threadIdx.x & 31) == 0) flag_status(status, PA_DEV_WAIT_TIMEOUT);
    }
    return ok;
}

// The same for one thread (the MMA issuer).
__device__ __forceinline__ bool pf_wait1(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag, int32_t* status) {
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity, kWaitLimitNs, abort_flag)) return true;
    *abort_flag = 1;
    flag_status(status, PA_DEV_WAIT_TIMEOUT);
    return false;
}

// Producer warp: stage k holds keys [64 k, 64 k + 64): the segment's blocks 64 k / BS .. of K and
// V, each block as D / 64 boxes of BS rows x 128 bytes.  Blocks past the last needed one are not
// loaded (the stage's byte count follows); their rows lie past every query's position.
template <int D, int BS>
__device__ __forceinline__ void pf_produce(const PrefillParams& p, const CUtensorMap* tk, const CUtensorMap* tv, int b,
                                           int g, int nblk, int nst, uint32_t ring_s, const PfBars& bars,
                                           volatile int32_t* abort_flag, int lane) {
    using L = PfLayout<D, BS>;
    constexpr int BPS = L::kBlocksPerStage;
    if (lane == 0) {
        prefetch_tensormap(tk);
        prefetch_tensormap(tv);
    }
    const uint64_t policy = policy_evict_last();
    const int32_t* tab = p.block_tables + (size_t)b * p.max_blocks_per_seq;
    int issued = 0;
    int32_t blk = 0;
    for (int k = 0; k < nst; ++k) {
        const int jb0 = k * BPS;  // first block of the stage
        if ((jb0 & 31) == 0) blk = jb0 + lane < nblk ? __ldg(tab + jb0 + lane) : 0;  // 32 table entries at a time
        const int s = k % kPfStages;
        if (!pf_wait(bars.kv_empty(s), ((k / kPfStages) & 1) ^ 1, abort_flag, p.status)) break;
        const int nb = min(BPS, nblk - jb0);
        int32_t bids[BPS];
#pragma unroll
        for (int t = 0; t < BPS; ++t) {
            int32_t bid = __shfl_sync(0xffffffffu, blk, (jb0 + t) & 31);
            if (t < nb && (bid < 0 || bid >= p.num_blocks)) {  // warp-uniform
                if (lane == 0) flag_status(p.status, PA_DEV_BAD_BLOCK_ID);
                bid = 0;
            }
            bids[t] = bid;
        }
        if (lane == 0) {
            mbar_arrive_expect_tx(bars.kv_full(s), (uint32_t)(nb * BS * 128 * L::kPanels * 2));
            const uint32_t kdst = ring_s + s * L::kStageBytes, vdst = kdst + L::kKPBytes;
#pragma unroll
            for (int t = 0; t < BPS; ++t) {
                if (t < nb) {
                    const int32_t y = (bids[t] * p.num_kv_heads + g) * BS;
#pragma unroll
                    for (int pn = 0; pn < L::kPanels; ++pn) {
                        const uint32_t off = pn * L::kKVPanel + t * BS * 128;
                        tma_load_2d(kdst + off, tk, pn * 64, y, bars.kv_full(s), policy);
                        tma_load_2d(vdst + off, tv, pn * 64, y, bars.kv_full(s), policy);
                    }
                }
            }
        }
        issued = k + 1;
    }
    // never leave the CTA with copies still landing in its shared memory
    for (int kk = issued > kPfStages ? issued - kPfStages : 0; kk < issued; ++kk)
        mbar_wait(bars.kv_full(kk % kPfStages), (kk / kPfStages) & 1);
}

// MMA issuer (one thread).  S_{k+1} is issued before waiting for P_k, so the tensor core computes
// the next scores while the softmax works on this stage.
template <int D, int BS>
__device__ __forceinline__ void pf_mma(const PrefillParams& p, int nst, uint32_t q_s, uint32_t ring_s, uint32_t tmem,
                                       const PfBars& bars, volatile int32_t* abort_flag) {
    using L = PfLayout<D, BS>;
    constexpr uint32_t idesc_s = umma_idesc_bf16(kPfRows, kPfKeys, 0, 0);  // Q (K-major) x K^T (K-major)
    constexpr uint32_t idesc_o = umma_idesc_bf16(kPfRows, D, 0, 1);         // P (K-major) x V (MN-major)
    auto issue_s = [&](int k) {
        const int s = k % kPfStages;
        const uint32_t kst = ring_s + s * L::kStageBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint64_t a = umma_smem_desc(q_s + (ks >> 2) * L::kQPanel + (ks & 3) * 32, 16, 1024);
            const uint64_t bd = umma_smem_desc(kst + (ks >> 2) * L::kKVPanel + (ks & 3) * 32, 16, 1024);
            umma_bf16(tmem + kPfTmemS + kPfKeys * s, a, bd, idesc_s, ks > 0);
        }
        umma_commit(bars.s_full(s));
    };
    bool ok = pf_wait1(bars.q_ready(), 0, abort_flag, p.status) &&
              pf_wait1(bars.kv_full(0), 0, abort_flag, p.status);
    if (ok) {
        tc_fence_after();
        issue_s(0);
    }
    for (int k = 0; ok && k < nst; ++k) {
        if (k + 1 < nst) {
            const int s1 = (k + 1) % kPfStages, ph = ((k + 1) / kPfStages) & 1;
            ok = pf_wait1(bars.kv_full(s1), ph, abort_flag, p.status) &&
                 pf_wait1(bars.s_free(s1), ph ^ 1, abort_flag, p.status);
            if (!ok) break;
            tc_fence_after();
            issue_s(k + 1);
        }
        const int s = k % kPfStages;
        if (!pf_wait1(bars.p_ready(s), (k / kPfStages) & 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t pst = ring_s + s * L::kStageBytes, vst = pst + L::kKPBytes;
#pragma unroll
        for (int kk = 0; kk < kPfKeys / 16; ++kk) {
            const uint64_t a = umma_smem_desc(pst + kk * 32, 16, 1024);
            const uint64_t bd = umma_smem_desc(vst + kk * 16 * 128, L::kKVPanel, 1024);
            umma_bf16(tmem, a, bd, idesc_o, (k > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bars.kv_empty(s));  // the stage may be refilled
        umma_commit(bars.o_done());
        if (k == nst - 1) umma_commit(bars.o_final());
    }
    // every MMA issued has completed before the CTA may free TMEM or its shared memory
    umma_commit(bars.mma_drain());
    mbar_wait(bars.mma_drain(), 0);
}

// Softmax warp w (0..3): query row r = 32 w + lane of the tile, TMEM lane r.
template <int D, int BS>
__device__ __forceinline__ void pf_softmax(const PrefillParams& p, int b, int g, int c0, int n, int len, int i0, int i1,
                                           int nst, uint8_t* base, uint32_t base_s, uint32_t tmem, const PfBars& bars,
                                           volatile int32_t* abort_flag, int warp, int lane) {
    using L = PfLayout<D, BS>;
    const int G = p.group, Hq = p.num_q_heads;
    const int rows_used = p.tile_tokens * G;
    const int r = 32 * warp + lane;
    const int tok = i0 + r / G;
    const bool valid = r < rows_used && tok < i1;
    const int pos_last = len - n + i1 - 1;
    // padding rows take the tile's last position: their scores stay finite and they are never stored
    const int pos = valid ? len - n + tok : pos_last;
    const int nkeys = pos_last + 1;
    const uint32_t lane_tmem = tmem + ((uint32_t)(32 * warp) << 16);

    // ---- Q row r into the swizzled K-major tile ----
    {
        const size_t qrow = ((size_t)(c0 + (valid ? tok : i0)) * Hq + (size_t)g * G + r % G) * D;
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) + qrow);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            const uint4 v = valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(base + L::kQOff + (c >> 3) * L::kQPanel + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
        }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars.q_ready());

    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int k = 0; k < nst; ++k) {
        const int s = k % kPfStages, ph = (k / kPfStages) & 1;
        if (!pf_wait(bars.s_full(s), ph, abort_flag, p.status)) {
            ok = false;
            break;
        }
        tc_fence_after();
        uint32_t sv0[32], sv1[32];
        tmem_ld32(lane_tmem + kPfTmemS + kPfKeys * s, sv0);
        tmem_ld32(lane_tmem + kPfTmemS + kPfKeys * s + 32, sv1);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.s_free(s));

        // base-2 scores with the causal mask: key t is visible to the row at position pos iff t <= pos
        const int key0 = k * kPfKeys;
        float x[kPfKeys];
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kPfKeys; ++c) {
            x[c] = key0 + c <= pos ? __uint_as_float(c < 32 ? sv0[c] : sv1[c - 32]) * p.scale_log2 : -INFINITY;
            mx = fmaxf(mx, x[c]);
        }
        const float m_new = fmaxf(m_run, mx);  // finite: stage 0 holds key 0, which every row sees
        if (k == 0) {
            m_run = m_new;
        } else {
            const bool need = m_new > m_run + kPfRescaleLog2;
            if (__any_sync(0xffffffffu, need)) {
                // O holds P V of the earlier stages: rescale it in TMEM once P_{k-1} V_{k-1} is done.
                // S_k was issued after P_{k-2} V_{k-2}, so that one has completed, and P_k V_k waits
                // for this warp: the phase of parity k - 1 is the one in progress or just completed.
                if (!pf_wait(bars.o_done(), (k - 1) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float f = need ? fast_exp2(m_run - m_new) : 1.f;
#pragma unroll
                for (int c0o = 0; c0o < D; c0o += 32) {
                    uint32_t ov[32];
                    tmem_ld32(lane_tmem + c0o, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
                    tmem_st32(lane_tmem + c0o, ov);
                }
                tmem_wait_st();
                if (need) {
                    l_run *= f;
                    m_run = m_new;
                }
            }
        }
        // P row r (bf16) over the stage's K, which S_k has finished reading; the sum uses the
        // rounded weights that P V uses
        uint8_t* pst = base + L::kRingOff + s * L::kStageBytes;
        float sum = 0.f;
#pragma unroll
        for (int c8 = 0; c8 < kPfKeys / 8; ++c8) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                w[e] = pack_bf16x2(fast_exp2(x[8 * c8 + 2 * e] - m_run), fast_exp2(x[8 * c8 + 2 * e + 1] - m_run));
                sum += bf16_lo(w[e]) + bf16_hi(w[e]);
            }
            *reinterpret_cast<uint4*>(pst + r * 128 + ((c8 ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        l_run += sum;
        // V rows past the tile's last position carry zero weight in every row, but their slots may
        // hold any bits (unfilled slots, or rows no block was loaded into): zero them
        const int vlim = nkeys - key0;
        if (vlim < kPfKeys) {
            if (!pf_wait(bars.kv_full(s), ph, abort_flag, p.status)) {
                ok = false;
                break;
            }
            uint8_t* vst = pst + L::kKPBytes;
            const int nz = (kPfKeys - vlim) * 8 * L::kPanels;  // 16-byte chunks to clear
            for (int i = r; i < nz; i += kPfRows) {
                const int pn = i / ((kPfKeys - vlim) * 8), rem = i - pn * ((kPfKeys - vlim) * 8);
                *reinterpret_cast<uint4*>(vst + pn * L::kKVPanel + (vlim + rem / 8) * 128 + (rem & 7) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.p_ready(s));
    }
    if (!ok || !pf_wait(bars.o_final(), 0, abort_flag, p.status)) return;
    tc_fence_after();

    // ---- O / l from TMEM to out (bf16) ----
    const float inv = 1.f / l_run;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                          ((size_t)(c0 + (valid ? tok : i0)) * Hq + (size_t)g * G + r % G) * D);
#pragma unroll
    for (int c0o = 0; c0o < D; c0o += 32) {
        uint32_t ov[32];
        tmem_ld32(lane_tmem + c0o, ov);
        tmem_wait_ld();
        if (valid) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = pack_bf16x2(__uint_as_float(ov[8 * q4 + 2 * e]) * inv, __uint_as_float(ov[8 * q4 + 2 * e + 1]) * inv);
                dst[c0o / 8 + q4] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
}

template <int D, int BS>
__global__ void __launch_bounds__(kPfThreads, kPfCtasPerSm) prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmap_k,
                                                             const __grid_constant__ CUtensorMap tmap_v) {
    using L = PfLayout<D, BS>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_s - raw_s);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // unit: sequence b, KV head g, query tile j (the tiles that end latest go first)
    const int b = blockIdx.z, g = blockIdx.y;
    const int j = (int)gridDim.x - 1 - (int)blockIdx.x;
    const int c0 = __ldg(p.cu_q_lens + b), n = __ldg(p.cu_q_lens + b + 1) - c0;
    const int len = __ldg(p.seq_lens + b);
    const int i0 = j * p.tile_tokens;
    if (n <= 0 || i0 >= n) return;  // the whole CTA
    if (n > len || n > p.max_q_len || (int64_t)len > (int64_t)p.max_blocks_per_seq * BS || c0 < 0 ||
        (int64_t)c0 + n > p.num_q_tokens) {
        if (tid == 0 && j == 0 && g == 0) flag_status(p.status, PA_DEV_BAD_SEQ_LEN);
        return;
    }
    const int i1 = min(n, i0 + p.tile_tokens);
    const int nkeys = len - n + i1;                    // keys up to the tile's last position
    const int nblk = (nkeys + BS - 1) / BS;
    const int nst = (nkeys + kPfKeys - 1) / kPfKeys;   // 64-key stages

    volatile int32_t* misc = reinterpret_cast<volatile int32_t*>(base + L::kMiscOff);
    PfBars bars{base_s + L::kBarOff};
    if (tid == 0) {
        for (int s = 0; s < kPfStages; ++s) {
            mbar_init(bars.kv_full(s), 1);                  // the producer's expect_tx
            mbar_init(bars.kv_empty(s), 1);                 // tcgen05.commit after P V
            mbar_init(bars.s_full(s), 1);                   // tcgen05.commit after Q K^T
            mbar_init(bars.s_free(s), kPfSoftmaxWarps);     // each softmax warp has read its S rows
            mbar_init(bars.p_ready(s), kPfSoftmaxWarps);    // each softmax warp has written its P rows
        }
        mbar_init(bars.o_done(), 1);
        mbar_init(bars.o_final(), 1);
        mbar_init(bars.q_ready(), kPfSoftmaxWarps);
        mbar_init(bars.mma_drain(), 1);
        fence_barrier_init();
        misc[0] = 0;  // abort flag
    }
    if (warp == kPfMma) tmem_alloc(base_s + L::kMiscOff + 16, kPfTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base + L::kMiscOff + 16);

    if (warp == kPfProducer)
        pf_produce<D, BS>(p, &tmap_k, &tmap_v, b, g, nblk, nst, base_s + L::kRingOff, bars, misc, lane);
    else if (warp == kPfMma) {
        if (lane == 0) pf_mma<D, BS>(p, nst, base_s + L::kQOff, base_s + L::kRingOff, tmem, bars, misc);
        __syncwarp();
    } else
        pf_softmax<D, BS>(p, b, g, c0, n, len, i0, i1, nst, base, base_s, tmem, bars, misc, warp, lane);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kPfMma) tmem_dealloc(tmem, kPfTmemCols);
}

template <int D, int BS>
pa_status launch_prefill(const PrefillParams& p, const void* k_pool, const void* v_pool, int64_t rows, int num_seqs,
                         int max_q_len, cudaStream_t stream) {
    using L = PfLayout<D, BS>;
    int dev = 0, occ = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    const void* kfn = reinterpret_cast<const void*>(&prefill_kernel<D, BS>);
    if (!kernel_occupancy(dev, kfn, kPfThreads, L::kBytes, &occ)) return PA_ERR_CUDA;
    if (occ <= 0) return PA_ERR_UNSUPPORTED;
    CUtensorMap tk, tv;
    if (!pool_map(&tk, dev, k_pool, rows, D, BS, PA_BF16) || !pool_map(&tv, dev, v_pool, rows, D, BS, PA_BF16))
        return PA_ERR_CUDA;
    const dim3 grid((max_q_len + p.tile_tokens - 1) / p.tile_tokens, p.num_kv_heads, num_seqs);
    prefill_kernel<D, BS><<<grid, kPfThreads, L::kBytes, stream>>>(p, tk, tv);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_prefill_attention(void* out, const void* q, const void* k_pool, const void* v_pool,
                                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                                          const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t num_seqs,
                                          int32_t num_q_tokens, int32_t max_q_len, int32_t num_q_heads,
                                          int32_t num_kv_heads,
                                          int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
                                          pa_dtype dtype, int32_t* dev_status, void* stream) {
    if (dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads || max_q_len < 0 ||
        num_q_tokens < 0 ||
        max_blocks_per_seq <= 0 || num_blocks <= 0 || !std::isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (num_q_heads / num_kv_heads > 8 || (head_dim != 64 && head_dim != 128) || (block_size != 16 && block_size != 32) ||
        num_seqs > 65535 || num_kv_heads > 65535)
        return PA_ERR_UNSUPPORTED;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens || !cu_q_lens) return PA_ERR_INVALID_ARG;
    auto a16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
    auto a4 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; };
    if (!a16(out) || !a16(q) || !a16(k_pool) || !a16(v_pool) || !a4(block_tables) || !a4(seq_lens) || !a4(cu_q_lens) ||
        !a4(dev_status))
        return PA_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)num_blocks * num_kv_heads * block_size;
    if (rows >= INT32_MAX) return PA_ERR_UNSUPPORTED;
    if (max_q_len == 0 || num_q_tokens == 0) return PA_OK;
    if ((int64_t)num_q_tokens * num_q_heads * head_dim >= INT32_MAX * 2ll) return PA_ERR_UNSUPPORTED;
    PrefillParams p;
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.cu_q_lens = cu_q_lens;
    p.status = dev_status;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.num_blocks = num_blocks;
    p.group = num_q_heads / num_kv_heads;
    p.tile_tokens = kPfRows / p.group;
    p.num_q_tokens = num_q_tokens;
    p.max_q_len = max_q_len;
    p.scale_log2 = scale * 1.4426950408889634f;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (head_dim == 128 && block_size == 16) return launch_prefill<128, 16>(p, k_pool, v_pool, rows, num_seqs, max_q_len, st);
    if (head_dim == 128 && block_size == 32) return launch_prefill<128, 32>(p, k_pool, v_pool, rows, num_seqs, max_q_len, st);
    if (head_dim == 64 && block_size == 16) return launch_prefill<64, 16>(p, k_pool, v_pool, rows, num_seqs, max_q_len, st);
    return launch_prefill<64, 32>(p, k_pool, v_pool, rows, num_seqs, max_q_len, st);
}
