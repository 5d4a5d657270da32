// Host side of pa_decode_attention: argument checks, the workspace layout,
// grid sizing, the TMA descriptors of the two pools, and the launch.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <mutex>
#include <vector>

#include "pa_internal.h"
#include "pa_plan.h"

namespace pa {
namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_ctas_per_sm{0};  // 0 = the per-path default
std::atomic<uint64_t> g_wait_limit_ns{0};  // 0 = kWaitLimitNs
std::atomic<int> g_merge_mode{0};          // 0 = chosen per launch, 1 = in the decode kernel, 2 = merge_kernel
std::atomic<int> g_seg_units{0};           // 0 = the compute path's weight of a segment, else this many units
std::atomic<int> g_wave_skew{-1};          // -1 = the compute path's skew of the CTA shares, else this one

struct DeviceInfo {
    int sms = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

bool current_device(int* dev, int* sms) {
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_dev[*dev].sms == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess || n <= 0) return false;
        g_dev[*dev].sms = n;
    }
    *sms = g_dev[*dev].sms;
    return true;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D view of a pool: rows = num_blocks * Hkv * BS, columns = head_dim; one
// box = BS rows x 128 bytes, loaded with the 128-byte swizzle.
bool encode_pool_map(CUtensorMap* map, const void* pool, int64_t rows, int head_dim, int block_size, pa_dtype dt) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const int elem = dt == PA_F32 ? 4 : (dt == PA_BF16 ? 2 : 1);
    cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)head_dim * elem};
    cuuint32_t box[2] = {(cuuint32_t)(128 / elem), (cuuint32_t)block_size};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType ty = dt == PA_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : dt == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = enc(map, ty, 2,
                     const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

// The pool maps of recent calls: an encoded map depends only on the pool's
// address and shape, so serving loops that pass the same pools every step
// reuse it instead of encoding two maps per call.
struct PoolMapEntry {
    int dev;
    const void* pool;
    int64_t rows;
    int head_dim, block_size;
    pa_dtype dt;
    CUtensorMap map;
};
constexpr int kPoolMapCache = 16;
static PoolMapEntry g_maps[kPoolMapCache];
static int g_maps_used = 0, g_maps_next = 0;

bool pool_map(CUtensorMap* map, int dev, const void* pool, int64_t rows, int head_dim, int block_size, pa_dtype dt) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < g_maps_used; ++i) {
        const PoolMapEntry& e = g_maps[i];
        if (e.dev == dev && e.pool == pool && e.rows == rows && e.head_dim == head_dim &&
            e.block_size == block_size && e.dt == dt) {
            *map = e.map;
            return true;
        }
    }
    if (!encode_pool_map(map, pool, rows, head_dim, block_size, dt)) return false;
    PoolMapEntry& e = g_maps[g_maps_next];
    e = PoolMapEntry{dev, pool, rows, head_dim, block_size, dt, *map};
    g_maps_next = (g_maps_next + 1) % kPoolMapCache;
    if (g_maps_used < kPoolMapCache) ++g_maps_used;
    return true;
}

// Query rows of a prefill tile: q [tokens][heads][head_dim] bf16 as a 3-D tensor
// (head_dim, heads, tokens); one box = 64 elements (128 bytes, 128-byte swizzle)
// x box_heads heads x box_tokens tokens, i.e. box_heads * box_tokens rows of 128
// bytes in token-major order.  Out-of-range tokens read as zero.  Cached per
// (device, q, shape) like the pool maps.
struct QMapEntry {
    int dev;
    const void* q;
    int64_t tokens;
    int heads, head_dim, box_heads, box_tokens;
    CUtensorMap map;
};
static QMapEntry g_qmaps[kPoolMapCache];
static int g_qmaps_used = 0, g_qmaps_next = 0;

bool prefill_q_map(CUtensorMap* map, int dev, const void* q, int64_t tokens, int heads, int head_dim, int box_heads,
                   int box_tokens) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < g_qmaps_used; ++i) {
        const QMapEntry& e = g_qmaps[i];
        if (e.dev == dev && e.q == q && e.tokens == tokens && e.heads == heads && e.head_dim == head_dim &&
            e.box_heads == box_heads && e.box_tokens == box_tokens) {
            *map = e.map;
            return true;
        }
    }
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)heads, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)heads * head_dim * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)box_heads, (cuuint32_t)box_tokens};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    QMapEntry& e = g_qmaps[g_qmaps_next];
    e = QMapEntry{dev, q, tokens, heads, head_dim, box_heads, box_tokens, *map};
    g_qmaps_next = (g_qmaps_next + 1) % kPoolMapCache;
    if (g_qmaps_used < kPoolMapCache) ++g_qmaps_used;
    return true;
}

// Dynamic shared memory opted into, and the occupancy found, per (device,
// kernel, shared-memory size): set and queried once instead of every call.
struct KernelEntry {
    int dev;
    const void* kernel;
    int smem_attr;  // largest dynamic shared memory opted into so far
    int occ_smem;   // shared memory size of the cached occupancy
    int occ;
};
constexpr int kKernelCache = 128;
static KernelEntry g_kernels[kKernelCache];
static int g_kernels_used = 0;

bool kernel_occupancy(int dev, const void* kernel, int threads, int smem, int* occ) {
    std::lock_guard<std::mutex> lk(g_mu);
    KernelEntry* e = nullptr;
    for (int i = 0; i < g_kernels_used; ++i)
        if (g_kernels[i].dev == dev && g_kernels[i].kernel == kernel) e = &g_kernels[i];
    if (e && e->occ_smem == smem) {
        *occ = e->occ;
        return true;
    }
    if (!e || e->smem_attr < smem) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return false;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess) return false;
    if (!e && g_kernels_used < kKernelCache) e = &g_kernels[g_kernels_used++];
    if (e) {
        const int attr = e->kernel == kernel && e->dev == dev && e->smem_attr > smem ? e->smem_attr : smem;
        *e = KernelEntry{dev, kernel, attr, smem, n};
    }
    *occ = n;
    return true;
}

// Registers per thread of a kernel (cudaFuncGetAttributes), cached per kernel.
static bool kernel_regs(const void* kernel, int* regs) {
    static const void* keys[kKernelCache];
    static int vals[kKernelCache];
    static int used = 0;
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < used; ++i)
        if (keys[i] == kernel) {
            *regs = vals[i];
            return true;
        }
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, kernel) != cudaSuccess) return false;
    if (used < kKernelCache) {
        keys[used] = kernel;
        vals[used++] = a.numRegs;
    }
    *regs = a.numRegs;
    return true;
}

namespace {

struct WorkspaceLayout {
    size_t counts_off, partials_off, total;
};

// The status head, one merge counter per CTA (rounded up to 256 bytes), then two partial slots
// for each of `ctas` CTAs.
WorkspaceLayout workspace_layout(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int64_t ctas) {
    WorkspaceLayout w;
    const size_t G = (size_t)(num_q_heads / num_kv_heads);
    w.counts_off = kStatusHeadBytes;
    w.partials_off = w.counts_off + (((size_t)ctas * 4 + 255) & ~(size_t)255);
    w.total = w.partials_off + (size_t)2 * ctas * partial_slot_floats((int)G, head_dim) * 4;
    return w;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pa_status check_shapes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                       int32_t block_size) {
    if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0) return PA_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads) return PA_ERR_INVALID_ARG;
    if (num_q_heads / num_kv_heads > 8) return PA_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (block_size != 16 && block_size != 32) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

// Picks the compiled variant, the build and the grid for these shapes on the current device.
struct LaunchPlan {
    DecodeVariant v;
    bool mma;
    int smem;
    int grid;
    int sms;
    int stages;
    int threads;
    int merge_smem;
    int merge_grid;
    bool merge_in_kernel;
    int seg_units;  // the range balance's weight of a segment (DecodeParams::seg_units)
    int wave_skew;  // the CTA shares' skew by dispatch wave (DecodeParams::wave_skew)
};

pa_status plan_launch(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, int32_t max_tiles_per_head, bool fixed, pa_dtype dtype, LaunchPlan* lp) {
    int dev = 0;
    if (!current_device(&dev, &lp->sms)) return PA_ERR_CUDA;
    const int G = num_q_heads / num_kv_heads;
    // dtype is the pool's: PA_FP8_E4M3 pools pair with bf16 queries and always take the
    // tensor cores (their codes are widened in registers); bf16 does for 4+ query heads
    lp->mma = (dtype == PA_BF16 && G >= 4) || dtype == PA_FP8_E4M3;
    bool found = dtype == PA_F32         ? decode_variant_f32(head_dim, block_size, G, &lp->v)
                 : dtype == PA_FP8_E4M3 ? decode_variant_fp8(head_dim, block_size, G, &lp->v)
                 : lp->mma              ? decode_variant_bf16_mma(head_dim, block_size, &lp->v)
                                        : decode_variant_bf16_fma(head_dim, block_size, G, &lp->v);
    if (!found) return PA_ERR_UNSUPPORTED;
    // Default CTAs per SM: the bf16 tensor-core path, which spends little time per tile,
    // keeps four (about 128 KB of tiles in flight, enough to cover HBM latency with fewer
    // split points); the CUDA-core path and the FP8 tensor-core path (which widens every
    // stage first) take as many as fit.
    int want = g_ctas_per_sm.load();
    if (want <= 0) want = lp->mma && dtype == PA_BF16 ? kDefaultCtasPerSmMma : kMaxCtasPerSm;
    const int64_t tiles_bound = (int64_t)num_seqs * num_kv_heads * max_tiles_per_head;
    struct Shape {
        int smem, per_sm, grid;
    };
    auto shape_of = [&](const DecodeBuild& b, Shape* sh) -> pa_status {
        sh->smem = b.smem_bytes(num_seqs, fixed);
        if (sh->smem > kMaxSmem) return PA_ERR_UNSUPPORTED;
        int occ = 0;
        if (!kernel_occupancy(dev, b.kernel, b.threads, sh->smem, &occ)) return PA_ERR_CUDA;
        if (occ <= 0) return PA_ERR_UNSUPPORTED;
        sh->per_sm = occ < want ? occ : want;
        int64_t grid = (int64_t)lp->sms * sh->per_sm;
        if (grid > tiles_bound) grid = tiles_bound;
        sh->grid = (int)(grid < 1 ? 1 : grid);
        return PA_OK;
    };
    Shape in{}, mk{};
    pa_status st = shape_of(lp->v.in, &in);
    if (st == PA_OK) st = shape_of(lp->v.mk, &mk);
    if (st != PA_OK) return st;
    // the merge kernel (with the mk build): a group of min(32, G D / 16) lanes per CTA
    // boundary (at most one split segment each), at most one CTA per SM
    lp->merge_smem = merge_smem_bytes(num_seqs, fixed);
    if (lp->merge_smem > kMaxSmem) return PA_ERR_UNSUPPORTED;
    int mocc = 0;
    if (!kernel_occupancy(dev, lp->v.merge_kernel, kMergeThreads, lp->merge_smem, &mocc)) return PA_ERR_CUDA;
    if (mocc <= 0) return PA_ERR_UNSUPPORTED;
    const int lps = G * head_dim / 16 < 32 ? G * head_dim / 16 : 32;
    const int64_t groups_per_cta = (kMergeThreads / 32) * (32 / lps);
    const int64_t merge_ctas = (mk.grid - 1 + groups_per_cta - 1) / groups_per_cta;
    lp->merge_grid = (int)(merge_ctas < 1 ? 1 : merge_ctas < lp->sms ? merge_ctas : lp->sms);
    // Where split segments are merged.  merge_kernel costs the decode CTAs nothing and
    // runs its plan while they stream, but only if one of its CTAs fits on an SM beside
    // the decode's (registers: 256 per warp granule; shared memory: 1 KB reserved per
    // CTA); it then merges right after the grid.  The in-kernel merge costs each split
    // piece a release fence and a count, and its merges run mid-range when CTAs hold
    // several segments each (the piece shared with the next CTA is walked first).  On
    // the HBM-bound paths (bf16) it takes over when segments outnumber CTAs 3:2, or when
    // merge_kernel could only start once decode CTAs exit.  Over FP8 pools the two
    // builds differ: the in-kernel one has one consumer warp per CTA and 8 CTAs per SM,
    // the merge-kernel one three consumer warps per CTA (the consumer is the bound, and
    // its fence and count stall the only consumer warp); with segments weighted as FP8
    // ranges weigh them the second is faster on every workload measured, though its four
    // CTAs fill an SM's registers and merge_kernel starts only as they exit, so FP8 calls
    // always take it.  With fixed partitions
    // (long contexts) a segment spans many CTAs and is merged after the streaming either
    // way: merge_kernel.  (Measured on GB300 on the workloads of the pages: each rule
    // picked the faster choice or one within 0.5 % of it.)
    int dregs = 0, mregs = 0;
    if (!kernel_regs(lp->v.mk.kernel, &dregs) || !kernel_regs(lp->v.merge_kernel, &mregs)) return PA_ERR_CUDA;
    auto warp_regs = [](int r) { return (int64_t)(r * 32 + 255) / 256 * 256; };
    const int64_t regs_used = (int64_t)mk.per_sm * (lp->v.mk.threads / 32) * warp_regs(dregs);
    const bool merge_fits = regs_used + (kMergeThreads / 32) * warp_regs(mregs) <= 65536 &&
                            (int64_t)mk.per_sm * (mk.smem + 1024) + lp->merge_smem + 1024 <= 228 * 1024;
    const int64_t segments = (int64_t)num_seqs * num_kv_heads;
    const int mode = g_merge_mode.load();
    const bool auto_in_kernel = dtype != PA_FP8_E4M3 && (2 * segments >= 3 * in.grid || !merge_fits);
    lp->merge_in_kernel = lp->v.merge_in_kernel_ok && (mode == 1 || (mode == 0 && !fixed && auto_in_kernel));
    const DecodeBuild& b = lp->merge_in_kernel ? lp->v.in : lp->v.mk;
    const Shape& sh = lp->merge_in_kernel ? in : mk;
    const int su = g_seg_units.load();
    lp->seg_units = su > 0                     ? su
                    : dtype == PA_FP8_E4M3     ? PA_SEG_UNITS_FP8
                    : lp->mma                  ? PA_SEG_UNITS_MMA
                                               : PA_SEG_UNITS_FMA;
    const int ws = g_wave_skew.load();
    lp->wave_skew = ws >= 0 ? ws : dtype == PA_FP8_E4M3 ? PA_WAVE_SKEW_FP8 : 0;
    lp->smem = sh.smem;
    lp->grid = sh.grid;
    lp->stages = b.stages;
    lp->threads = b.threads;
    return PA_OK;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                               int32_t head_dim, size_t* bytes_out) {
    if (!bytes_out) return PA_ERR_INVALID_ARG;
    if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || num_q_heads % num_kv_heads)
        return PA_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (!current_device(&dev, &sms)) return PA_ERR_CUDA;
    // enough for the largest grid any launch on this device can take
    *bytes_out = workspace_layout(num_q_heads, num_kv_heads, head_dim, (int64_t)sms * kMaxCtasPerSm).total;
    return PA_OK;
}

extern "C" pa_status pa_decode_set_ctas_per_sm(int32_t ctas) {
    if (ctas < 0 || ctas > kMaxCtasPerSm) return PA_ERR_INVALID_ARG;
    g_ctas_per_sm.store(ctas);
    return PA_OK;
}

extern "C" pa_status pa_debug_set_merge_mode(int32_t mode) {
    if (mode < 0 || mode > 2) return PA_ERR_INVALID_ARG;
    g_merge_mode.store(mode);
    return PA_OK;
}

extern "C" pa_status pa_debug_set_seg_units(int32_t units) {
    if (units < 0 || units > kMaxSegUnits) return PA_ERR_INVALID_ARG;
    g_seg_units.store(units);
    return PA_OK;
}

extern "C" pa_status pa_debug_plan_ranges(const int32_t* block_counts, int32_t num_seqs, int32_t num_kv_heads,
                                          int32_t partition_tiles, int32_t seg_units, int32_t num_ctas,
                                          int32_t wave_ctas, int32_t wave_skew, int64_t* starts_out,
                                          int32_t* owners_out, size_t owners_cap, int32_t* working_ctas_out) {
    if (!block_counts || !starts_out || !working_ctas_out || num_seqs <= 0 || num_kv_heads <= 0 ||
        partition_tiles < 0 || seg_units < 0 || seg_units > kMaxSegUnits || num_ctas <= 0 || wave_ctas <= 0 ||
        wave_skew < 0 || wave_skew > kWaveWeight / 8)
        return PA_ERR_INVALID_ARG;
    std::vector<int32_t> pref(num_seqs + 1), upref(num_seqs + 1);
    int64_t nb = 0, np = 0;
    for (int b = 0; b < num_seqs; ++b) {
        if (block_counts[b] < 0) return PA_ERR_INVALID_ARG;
        pref[b] = (int32_t)nb;
        upref[b] = (int32_t)np;
        nb += block_counts[b];
        if (partition_tiles > 0) np += (block_counts[b] + partition_tiles - 1) / partition_tiles;
        if (nb * num_kv_heads >= (int64_t)1 << 31) return PA_ERR_INVALID_ARG;
    }
    pref[num_seqs] = (int32_t)nb;
    upref[num_seqs] = (int32_t)np;
    const Plan P = plan_from_prefix(pref.data(), upref.data(), num_seqs, num_kv_heads, partition_tiles, seg_units,
                                    num_ctas, wave_ctas, wave_skew);
    if (owners_out && owners_cap < (size_t)P.T) return PA_ERR_WORKSPACE_TOO_SMALL;
    *working_ctas_out = P.C;
    for (int c = 0; c <= P.C; ++c) {
        int64_t split = -1;
        int seq = 0;
        starts_out[c] = P.T > 0 ? P.cta_start(c, &split, &seq) : 0;
    }
    if (owners_out)
        for (int64_t t = 0; t < P.T; ++t) owners_out[t] = P.cta_of(t);
    return PA_OK;
}

extern "C" pa_status pa_debug_set_wave_skew(int32_t skew) {
    if (skew < -1 || skew > kWaveWeight / 8) return PA_ERR_INVALID_ARG;
    g_wave_skew.store(skew);
    return PA_OK;
}

extern "C" pa_status pa_debug_set_wait_limit_ns(uint64_t ns) {
    if (ns > kWaitLimitNs) return PA_ERR_INVALID_ARG;
    g_wait_limit_ns.store(ns);
    return PA_OK;
}

extern "C" pa_status pa_decode_launch_info(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                           int32_t head_dim, int32_t block_size, int32_t max_blocks_per_seq,
                                           int32_t partition_tokens, pa_dtype dtype, int32_t* ctas,
                                           int32_t* stages, int32_t* smem_bytes, int32_t* uses_mma) {
    if (dtype != PA_F32 && dtype != PA_BF16 && dtype != PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;
    pa_status s = check_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size);
    if (s != PA_OK) return s;
    if (max_blocks_per_seq <= 0 || partition_tokens < 0 || partition_tokens % block_size) return PA_ERR_INVALID_ARG;
    LaunchPlan lp;
    s = plan_launch(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                    partition_tokens > 0, dtype, &lp);
    if (s != PA_OK) return s;
    if (ctas) *ctas = lp.grid;
    if (stages) *stages = lp.stages;
    if (smem_bytes) *smem_bytes = lp.smem;
    if (uses_mma) *uses_mma = lp.mma ? 1 : 0;
    return PA_OK;
}

extern "C" pa_status pa_decode_kernels_per_call(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                                int32_t head_dim, int32_t block_size, int32_t max_blocks_per_seq,
                                                int32_t partition_tokens, pa_dtype dtype, int32_t* kernels) {
    if (dtype != PA_F32 && dtype != PA_BF16 && dtype != PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;
    if (!kernels) return PA_ERR_INVALID_ARG;
    pa_status s = check_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size);
    if (s != PA_OK) return s;
    if (max_blocks_per_seq <= 0 || partition_tokens < 0 || partition_tokens % block_size) return PA_ERR_INVALID_ARG;
    LaunchPlan lp;
    s = plan_launch(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                    partition_tokens > 0, dtype, &lp);
    if (s != PA_OK) return s;
    *kernels = lp.merge_in_kernel ? 1 : 2;
    return PA_OK;
}

namespace pa {

// Shared by pa_decode_attention (pools of the query dtype),
// pa_decode_attention_fp8 (FP8 pools, bf16 queries, K and V scales) and the
// static-workspace entry point (clear_status: zero the status head on the
// stream once every check has passed, right before the launch).
pa_status decode_common(void* out, const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
                        int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t max_seq_len, int32_t num_seqs,
                        int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                        int32_t num_blocks, float scale, int32_t partition_tokens, void* workspace,
                        size_t workspace_bytes, pa_dtype dtype, float k_scale, float v_scale, void* stream,
                        bool clear_status, const void* plan, size_t plan_bytes) {
    if (dtype != PA_F32 && dtype != PA_BF16 && dtype != PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;
    pa_status s = check_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size);
    if (s != PA_OK) return s;
    if (dtype == PA_FP8_E4M3 && head_dim != 128) return PA_ERR_UNSUPPORTED;  // a pool row fills one 128-byte panel
    if (!std::isfinite(k_scale) || !std::isfinite(v_scale) || !(k_scale > 0.f) || !(v_scale > 0.f))
        return PA_ERR_INVALID_ARG;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens || !workspace) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return PA_ERR_INVALID_ARG;
    if (max_blocks_per_seq <= 0 || num_blocks <= 0 || max_seq_len < 0) return PA_ERR_INVALID_ARG;
    if (partition_tokens < 0 || (partition_tokens % block_size) != 0) return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)num_blocks * num_kv_heads * block_size;
    const int64_t tiles = (int64_t)num_seqs * num_kv_heads * max_blocks_per_seq;
    if (rows >= INT32_MAX || tiles >= INT32_MAX || (int64_t)num_seqs * num_q_heads * head_dim >= INT32_MAX)
        return PA_ERR_UNSUPPORTED;

    const int64_t table_len = (int64_t)max_blocks_per_seq * block_size;
    const int32_t max_len = (int32_t)(max_seq_len < table_len ? max_seq_len : table_len);
    const int32_t max_tiles = (max_len + block_size - 1) / block_size;
    const bool fixed = partition_tokens > 0;
    LaunchPlan lp;
    s = plan_launch(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_tiles > 0 ? max_tiles : 1, fixed,
                    dtype, &lp);
    if (s != PA_OK) return s;
    // the bytes this launch touches: the status head, a merge counter and two partial slots per CTA of its grid
    const WorkspaceLayout wl = workspace_layout(num_q_heads, num_kv_heads, head_dim, lp.grid);
    if (workspace_bytes < wl.total) return PA_ERR_WORKSPACE_TOO_SMALL;
    if (plan && ((reinterpret_cast<uintptr_t>(plan) & 3u) || plan_bytes < (size_t)plan_words(num_seqs, lp.grid) * 4))
        return PA_ERR_INVALID_ARG;

    CUtensorMap tk, tv;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (!pool_map(&tk, dev, k_pool, rows, head_dim, block_size, dtype) ||
        !pool_map(&tv, dev, v_pool, rows, head_dim, block_size, dtype))
        return PA_ERR_CUDA;

    DecodeParams p;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.status = reinterpret_cast<int32_t*>(ws);
    p.merge_counts = reinterpret_cast<int32_t*>(ws + wl.counts_off);
    p.partials = reinterpret_cast<float*>(ws + wl.partials_off);
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.max_len = max_len;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.num_blocks = num_blocks;
    p.group = num_q_heads / num_kv_heads;
    p.partition_tiles = partition_tokens / block_size;
    p.num_ctas = lp.grid;
    p.seg_units = lp.seg_units;
    p.wave_ctas = lp.sms;
    p.wave_skew = lp.wave_skew;
    p.scale_log2 = scale * 1.4426950408889634f * k_scale;
    p.out_scale = v_scale;
    const uint64_t lim = g_wait_limit_ns.load();
    p.wait_limit_ns = lim ? lim : kWaitLimitNs;
    p.merge_in_kernel = lp.merge_in_kernel ? 1 : 0;
    p.plan = static_cast<const int32_t*>(plan);
    if (clear_status && cudaMemsetAsync(workspace, 0, wl.partials_off, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PA_ERR_CUDA;
    lp.v.launch(p, tk, tv, lp.grid, lp.smem, lp.merge_grid, lp.merge_smem, static_cast<cudaStream_t>(stream));
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa

extern "C" pa_status pa_decode_attention(void* out, const void* q, const void* k_pool, const void* v_pool,
                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                         const int32_t* seq_lens, int32_t max_seq_len, int32_t num_seqs,
                                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                         int32_t block_size, int32_t num_blocks, float scale, int32_t partition_tokens,
                                         void* workspace, size_t workspace_bytes, pa_dtype dtype, void* stream) {
    if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    return pa::decode_common(out, q, k_pool, v_pool, block_tables, max_blocks_per_seq, seq_lens, max_seq_len, num_seqs,
                             num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, partition_tokens,
                             workspace, workspace_bytes, dtype, 1.f, 1.f, stream, false);
}

extern "C" pa_status pa_decode_attention_fp8(void* out, const void* q, const void* k_pool, const void* v_pool,
                                             float k_scale, float v_scale, const int32_t* block_tables,
                                             int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                             int32_t max_seq_len, int32_t num_seqs, int32_t num_q_heads,
                                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                             int32_t num_blocks, float scale, int32_t partition_tokens,
                                             void* workspace, size_t workspace_bytes, void* stream) {
    return pa::decode_common(out, q, k_pool, v_pool, block_tables, max_blocks_per_seq, seq_lens, max_seq_len, num_seqs,
                             num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, partition_tokens,
                             workspace, workspace_bytes, PA_FP8_E4M3, k_scale, v_scale, stream, false);
}

namespace {

// The launch a decode call with these arguments makes: its length bound, plan and grid.
pa_status decode_shape(int32_t max_blocks_per_seq, int32_t max_seq_len, int32_t num_seqs, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t partition_tokens,
                       pa_dtype dtype, int32_t* max_len_out, LaunchPlan* lp) {
    if (dtype != PA_F32 && dtype != PA_BF16 && dtype != PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;
    pa_status s = check_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size);
    if (s != PA_OK) return s;
    if (dtype == PA_FP8_E4M3 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (max_blocks_per_seq <= 0 || max_seq_len < 0) return PA_ERR_INVALID_ARG;
    if (partition_tokens < 0 || (partition_tokens % block_size) != 0) return PA_ERR_INVALID_ARG;
    if ((int64_t)num_seqs * num_kv_heads * max_blocks_per_seq >= INT32_MAX) return PA_ERR_UNSUPPORTED;
    const int64_t table_len = (int64_t)max_blocks_per_seq * block_size;
    const int32_t max_len = (int32_t)(max_seq_len < table_len ? max_seq_len : table_len);
    const int32_t max_tiles = (max_len + block_size - 1) / block_size;
    *max_len_out = max_len;
    return plan_launch(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_tiles > 0 ? max_tiles : 1,
                       partition_tokens > 0, dtype, lp);
}

}  // namespace

extern "C" pa_status pa_decode_plan_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t block_size, int32_t max_blocks_per_seq,
                                          int32_t max_seq_len, int32_t partition_tokens, pa_dtype dtype,
                                          size_t* bytes_out) {
    if (!bytes_out) return PA_ERR_INVALID_ARG;
    int32_t max_len = 0;
    LaunchPlan lp;
    pa_status s = decode_shape(max_blocks_per_seq, max_seq_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                               block_size, partition_tokens, dtype, &max_len, &lp);
    if (s != PA_OK) return s;
    *bytes_out = (size_t)plan_words(num_seqs, lp.grid) * 4;
    return PA_OK;
}

extern "C" pa_status pa_decode_build_plan(const int32_t* block_tables, int32_t max_blocks_per_seq,
                                          const int32_t* seq_lens, int32_t max_seq_len, int32_t num_seqs,
                                          int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                          int32_t block_size, int32_t partition_tokens, pa_dtype dtype,
                                          void* plan_out, size_t plan_bytes) {
    if (!block_tables || !seq_lens || !plan_out || (reinterpret_cast<uintptr_t>(plan_out) & 3u))
        return PA_ERR_INVALID_ARG;
    int32_t max_len = 0;
    LaunchPlan lp;
    pa_status s = decode_shape(max_blocks_per_seq, max_seq_len, num_seqs, num_q_heads, num_kv_heads, head_dim,
                               block_size, partition_tokens, dtype, &max_len, &lp);
    if (s != PA_OK) return s;
    const int B = num_seqs, Hkv = num_kv_heads, C = lp.grid;
    if (plan_bytes < (size_t)plan_words(B, C) * 4) return PA_ERR_WORKSPACE_TOO_SMALL;
    int32_t* pl = static_cast<int32_t*>(plan_out);
    const int PT = partition_tokens / block_size;
    const int A = lp.seg_units;
    for (int w = 0; w < kPlanHeaderWords; ++w) pl[w] = 0;
    pl[kPlanWMagic] = kPlanMagic;
    pl[kPlanWNumSeqs] = B;
    pl[kPlanWGrid] = C;
    pl[kPlanWKvHeads] = Hkv;
    pl[kPlanWPartitionTiles] = PT;
    pl[kPlanWSegUnits] = A;
    pl[kPlanWBlockSize] = block_size;
    pl[kPlanWMaxLen] = max_len;
    pl[kPlanWMergeInKernel] = lp.merge_in_kernel ? 1 : 0;
    pl[kPlanWMaxBlocks] = max_blocks_per_seq;
    pl[kPlanWWaveCtas] = lp.sms;
    pl[kPlanWWaveSkew] = lp.wave_skew;
    // the lengths scan of the kernels: clamped lengths, block and partition prefix sums
    int32_t* pref = pl + kPlanHeaderWords;
    int32_t* upref = pref + (B + 1);
    int32_t* lens = upref + (B + 1);
    int32_t nb_sum = 0, np_sum = 0;
    for (int b = 0; b < B; ++b) {
        const int len = clamp_len(seq_lens[b], max_len);
        const int nb = (len + block_size - 1) / block_size;
        lens[b] = len;
        pref[b] = nb_sum;
        upref[b] = PT > 0 ? np_sum : 0;
        nb_sum += nb;
        if (PT > 0) np_sum += (nb + PT - 1) / PT;
    }
    pref[B] = nb_sum;
    upref[B] = PT > 0 ? np_sum : 0;
    const Plan P = plan_from_prefix(pref, upref, B, Hkv, PT, A, C, lp.sms, lp.wave_skew);
    for (int c = 0; c < C; ++c) {
        int32_t* rec = pl + plan_rec_off(B, c);
        for (int w = 0; w < kPlanRecWords; ++w) rec[w] = 0;
        if (!(P.T > 0 && c < P.C)) {
            rec[kRecTa] = -1;
            continue;
        }
        int64_t s0 = -1, s1 = -1;
        int q0 = 0, q1 = 0;
        const int64_t t0 = P.cta_start(c, &s0, &q0), t1 = P.cta_start(c + 1, &s1, &q1);
        const int64_t ta = lp.merge_in_kernel ? s1 : -1;
        rec[kRecT0] = (int32_t)t0;
        rec[kRecT1] = (int32_t)t1;
        rec[kRecTa] = (int32_t)ta;
        rec[kRecSeq0] = q0;
        rec[kRecSeq1] = q1;
        // the table entries of the first (up to) 32 tiles of the range's first piece
        PieceIter<true> it;
        it.init(P, t0, t1, ta, q0, q1);
        int b = 0, h = 0, j0 = 0, j1 = 0;
        if (it.next(P, b, h, j0, j1)) {
            const int n = j1 - j0 < kPlanChunk ? j1 - j0 : kPlanChunk;
            for (int l = 0; l < n; ++l) rec[kRecFirst + l] = block_tables[(size_t)b * max_blocks_per_seq + j0 + l];
        }
    }
    return PA_OK;
}

extern "C" pa_status pa_decode_attention_planned(void* out, const void* q, const void* k_pool, const void* v_pool,
                                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                 const int32_t* seq_lens, int32_t max_seq_len, int32_t num_seqs,
                                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                                 int32_t block_size, int32_t num_blocks, float scale,
                                                 int32_t partition_tokens, void* workspace, size_t workspace_bytes,
                                                 pa_dtype dtype, const void* plan, size_t plan_bytes, void* stream) {
    if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (!plan) return PA_ERR_INVALID_ARG;
    return pa::decode_common(out, q, k_pool, v_pool, block_tables, max_blocks_per_seq, seq_lens, max_seq_len, num_seqs,
                             num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, partition_tokens,
                             workspace, workspace_bytes, dtype, 1.f, 1.f, stream, false, plan, plan_bytes);
}

extern "C" pa_status pa_decode_attention_fp8_planned(void* out, const void* q, const void* k_pool,
                                                     const void* v_pool, float k_scale, float v_scale,
                                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                     const int32_t* seq_lens, int32_t max_seq_len, int32_t num_seqs,
                                                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                                     int32_t block_size, int32_t num_blocks, float scale,
                                                     int32_t partition_tokens, void* workspace,
                                                     size_t workspace_bytes, const void* plan, size_t plan_bytes,
                                                     void* stream) {
    if (!plan) return PA_ERR_INVALID_ARG;
    return pa::decode_common(out, q, k_pool, v_pool, block_tables, max_blocks_per_seq, seq_lens, max_seq_len, num_seqs,
                             num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, partition_tokens,
                             workspace, workspace_bytes, PA_FP8_E4M3, k_scale, v_scale, stream, false, plan,
                             plan_bytes);
}
