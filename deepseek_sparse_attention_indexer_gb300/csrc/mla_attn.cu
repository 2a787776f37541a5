// mla_attn.cu -- sparse absorbed-MLA attention over the selected latent keys.
//
// What it computes (SlimServe "GLM52_PIPELINE_TRACE.md", section 6 "Attention
// core (absorbed MLA)"; exo PR #2539, sections "Prefill" and "Decode"): each
// query's 64 heads, 576 wide ([q_nope.wk_b 512 | q_pe 64]), attend over the
// query's selected rows of the shared latent cache ([kv_cmpr 512 | k_pe 64]):
//   s[h,t] = scale * q[h,:] . kv[idx_t,:],  p = softmax_t(s) in float32,
//   out[h,:] = sum_t p[h,t] * kv[idx_t, 0:512].
//
// How (GB300 design):
//   * Keys sit on the 128 TMEM lanes: S^T = K . Q^T (M = 128 gathered keys,
//     N = 64 heads, K = 576) and O^T = V^T . P^T (M = 128 latent dims, four
//     chunks, N = 64 heads, K = 128 keys).  Every MMA is a full-rate M = 128
//     tcgen05 MMA although the query has only 64 heads.
//   * The gathered tile is stored once, K-major with the 128-byte swizzle
//     (128 keys x 64 dims per 16 KB block, 9 blocks).  QK reads it K-major;
//     PV reads the very same bytes as the MN-major V^T operand, so the latent
//     rows are gathered once and used twice (keys and values).
//   * Sixteen worker warps do both the gather and the softmax.  A worker
//     warp copies 8 rows of a tile (four per 64-key half) with 16-byte
//     cp.async straight into the swizzled layout; one warp instruction copies
//     one 64-dim block of four different rows (8 lanes a row), so the L2
//     requests in flight spread over many rows rather than long spans of one
//     (measured: about twice the copy throughput of two-row spans).  PV runs
//     one 128-dim latent chunk at a time and frees that chunk's two blocks of
//     the stage as soon as it is consumed (the last chunk frees the P^T/rope
//     block too), so the next tile's copies of a chunk, and then its QK
//     segment, overlap the rest of PV (measured against releasing 64-key
//     halves: 1.93 -> 1.91 ms at 16k keys, 2.09 -> 1.91 ms at 64k keys).
//     The copies of tile t+1 are issued right after the warp's softmax of
//     tile t, so the whole CTA issues copies (cp.async throughput from L2
//     grows with the number of issuing warps).  QK waits per 128-dim chunk of
//     the K-dim.  Unselected or padding slots are zero-filled.  Above a
//     quarter of L2 of cache, each lane also prefetches into L2 the row it
//     copies one tile later.
//   * Two MMA-issuing warps: one issuing thread sustains an M128 N64 K16 MMA
//     only every ~70 cycles, two reach one every ~48 per SM.  Issuer i owns
//     latent chunks i and i + 2 (their QK into its own S^T partial sum, which
//     the softmax adds, and their PV); issuer 1 also the rope block.  The
//     issuing threads are instruction-bound, so each descriptor is a
//     precomputed base plus a compile-time offset on its low word.  What
//     bounds a tile is the shared-memory traffic of the operands and copies
//     plus the softmax between QK and PV: one 144 KB stage and the 72 KB Q^T
//     leave no room for a second tile or query to overlap it.
//   * Paged caches (PAGED): a row's cache address comes from the sequence's
//     page table, looked up after the index load.
//   * Softmax: four warps per TMEM lane quadrant, 16 heads each, one key per
//     thread.  Each head's reference maximum is taken from the query's first
//     tile (transposing warp butterfly + one shared-memory exchange); later
//     tiles only check, per thread, whether a score exceeds its reference by
//     more than 2^16, and only then reduce and rescale O^T in TMEM; the vote,
//     the reduction and the new references involve only the four warps (one
//     per lane quadrant) that share a group of 16 heads.
//     Numerator and denominator always share the reference, so the result is
//     the exact softmax.  P^T is written as bf16 into the (consumed) rope
//     block.
//   * The query's Q^T (72 KB) is loaded by TMA once per query.
//   * Decode splits a sequence's selected keys over CTAs and writes partial
//     (normalised output, lse) pairs; a small kernel merges them.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {

namespace {

constexpr int kH = DSA_HEADS;          // 64
constexpr int kD = DSA_QK_DIM;         // 576
constexpr int kDv = DSA_V_DIM;         // 512
constexpr int kRowBytes = kD * 2;      // 1152
constexpr int kTile = 128;             // keys per tile (MMA M)
constexpr int kBlkBytes = kTile * 128; // 16 KB: 128 keys x 64 dims
constexpr int kQBlkBytes = kH * 128;   // 8 KB: 64 heads x 64 dims
constexpr int kWorkerWarps = 16;                  // gather + softmax warps
constexpr int kWorkers = kWorkerWarps * 32;        // 512
constexpr int kIssuers = 2;                        // MMA-issuing warps
// Issuer i owns latent chunks i and i + 2 (their QK segments and their PV): interleaved, so that
// PV frees chunks 0 and 1 first, together, and the next tile's copies of them (issued in chunk
// order) start as early as they can.  Issuer 1 also runs the QK over the rope block.
constexpr int kMaxRegs = 96;                       // 19 warps: 5 share one 16K-register sub-partition
constexpr int kThreads = 32 * (1 + kIssuers) + kWorkers;  // warp 0 Q loader, warps 1-2 MMA, warps 3.. workers
constexpr int kHG = kH / (kWorkerWarps / 4);       // 16 heads per worker warp
constexpr int kGroupThreads = 4 * 32;              // the four warps sharing a head group
constexpr int kSegs = 4;               // PV releases the stage by 128-dim latent chunk (the rope block with the last)
static_assert(kWorkerWarps == 16 && kTile == 128, "a worker warp copies four rows of each 64-key half");
constexpr float kRescaleThreshold = 16.0f;  // log2 units
// m_neg (minus a head's reference maximum) before the reference is set: finite, so that a padding
// slot's -inf score still gives a -inf exponent (probability 0) while a valid score exceeds it
constexpr float kNoRef = 3.0e38f;

// smem layout (1024-aligned base)
constexpr int OFF_Q = 0;                               // 9 x 8 KB
constexpr int OFF_KV = OFF_Q + 9 * kQBlkBytes;         // 9 x 16 KB (block 8 = rope, then P^T)
constexpr int OFF_RED = OFF_KV + 9 * kBlkBytes;        // float [4][64]
constexpr int OFF_MNEG = OFF_RED + 4 * kH * 4;         // float [64]: minus the reference maxima
constexpr int OFF_ALPHA = OFF_MNEG + kH * 4;          // float [64]
constexpr int OFF_INVL = OFF_ALPHA + kH * 4;           // float [64]
constexpr int OFF_BAR = OFF_INVL + kH * 4;
// barriers: q_full, q_empty, seg_full[5], seg_free[4], s_full, p_full
constexpr int N_BARS = 2 + 5 + kSegs + 2;
constexpr int OFF_TMEM = OFF_BAR + N_BARS * 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int OFF_ITEM_T = OFF_ABORT + 4;              // int: the current item's tile count (workers)
constexpr int SMEM_BYTES = OFF_ITEM_T + 4 + 1024;

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;                       // S^T partial sums: issuer i's 64 columns at 64 i
constexpr uint32_t TM_O = 64 * kIssuers;           // O^T chunk c at TM_O + 64 c
static_assert(TM_O + 4 * 64 <= 512, "tensor memory columns");

constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 64, true, true);

struct AttnParams {
    const __nv_bfloat16* kv;   // [B][Nmax][576]
    const int32_t* idx;        // [rows][top_k]
    const int32_t* kv_len;     // [B] or nullptr (then every row may use Nmax keys)
    void* out;                 // final: [rows][64][512], float32 or bf16 (out_f32)
    int out_f32;               // 1: float32 output; 0: bf16 (round to nearest even)
    float* lse;                // final: [rows][64] or nullptr
    float* part_o;             // partial: [rows][nsplit][64][512]
    float* part_lse;           // partial: [rows][nsplit][64]
    int rows;                  // queries (prefill) or sequences (decode)
    int prefill;               // 1: all rows read batch 0 of kv; 0: row r reads batch r
    int Nmax;
    int top_k;
    int nsplit, split_len;     // slots per item = split_len (multiple of 128)
    int n_items;               // rows * nsplit
    float scale_log2;          // scale * log2(e)
    int32_t* status;           // device error word
    PageTable pages;           // paged cache (pages.table == nullptr: dense rows)
    int l2_prefetch;           // 1: prefetch each tile's cache rows into L2 one tile ahead (dense prefill)
};

// Waits of the worker warps (every lane polls).
__device__ __forceinline__ bool worker_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int32_t* status) {
    return mbar_wait(bar, parity, abort, status);
}

struct Item {
    int row, split, batch, slot0, slot_end, bound;
};

__device__ __forceinline__ Item decode_item(const AttnParams& p, int item) {
    Item it;
    it.row = item / p.nsplit;
    it.split = item % p.nsplit;
    it.batch = p.prefill ? 0 : it.row;
    it.slot0 = it.split * p.split_len;
    it.slot_end = min(p.top_k, it.slot0 + p.split_len);
    it.bound = p.kv_len ? min(__ldg(p.kv_len + it.batch), p.Nmax) : p.Nmax;
    return it;
}

__device__ __forceinline__ int nth_item(const AttnParams& p, int s) {
    int base = s * (int)gridDim.x;
    if (base >= p.n_items) return -1;
    int k = (s & 1) ? ((int)gridDim.x - 1 - (int)blockIdx.x) : (int)blockIdx.x;
    int item = base + k;
    return item < p.n_items ? item : -2;
}

// Number of 128-slot tiles up to the last non-negative index of the item's
// slot range (warp-collective; every lane gets the same answer).  A full
// selection ends with a valid index, so the last 32 slots are looked at first;
// otherwise (a query with fewer causal keys than top_k: a valid prefix, then
// -1) the range is scanned backwards 512 slots a round, 16 independent loads a
// lane, so that a short item costs a few L2 round trips rather than one per 32
// slots.
__device__ __forceinline__ int item_tiles(const AttnParams& p, const Item& I, uint32_t lane) {
    const int32_t* ir = p.idx + (int64_t)I.row * p.top_k;
    int hi = I.slot_end - 32;   // slots [hi, slot_end) first
    {
        const int s = hi + (int)lane;
        const bool v = (s >= I.slot0) && (s < I.slot_end) && (__ldg(ir + s) >= 0);
        const uint32_t m = __ballot_sync(0xffffffffu, v);
        if (m) return (hi + 31 - __clz(m) - I.slot0) / kTile + 1;
    }
    for (; hi > I.slot0; hi -= 512) {   // slots [max(slot0, hi - 512), hi)
        const int lo = hi - 512;
        int last = -1;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int s = lo + 32 * k + (int)lane;
            if (s >= I.slot0 && s < hi && __ldg(ir + s) >= 0) last = s;
        }
        last = __reduce_max_sync(0xffffffffu, last);
        if (last >= 0) return (last - I.slot0) / kTile + 1;
    }
    return 0;
}

// Transposing butterfly over a warp: on entry every lane holds 16 values (one
// per head of the warp's head group); on exit lanes 2i and 2i+1 hold the
// warp-wide reduction for head i of the group.
template <bool MAX>
__device__ __forceinline__ float warp_transpose_reduce16(const float (&x)[16], uint32_t lane) {
    float a[8];
    {
        const bool up = lane & 16;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float mine = up ? x[8 + k] : x[k];
            const float other = up ? x[k] : x[8 + k];
            const float recv = __shfl_xor_sync(0xffffffffu, other, 16);
            a[k] = MAX ? fmaxf(mine, recv) : mine + recv;
        }
    }
#pragma unroll
    for (int step = 0; step < 3; ++step) {
        const int half = 4 >> step;   // 4, 2, 1 values kept
        const int off = 8 >> step;    // shuffle distance 8, 4, 2
        const bool up = lane & off;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (k < half) {
                const float mine = up ? a[half + k] : a[k];
                const float other = up ? a[k] : a[half + k];
                const float recv = __shfl_xor_sync(0xffffffffu, other, off);
                a[k] = MAX ? fmaxf(mine, recv) : mine + recv;
            }
        }
    }
    const float o = __shfl_xor_sync(0xffffffffu, a[0], 1);
    return MAX ? fmaxf(a[0], o) : a[0] + o;
}


template <bool PARTIAL, bool PAGED>
__global__ void __maxnreg__(kMaxRegs)   // kThreads threads, one CTA per SM
    mla_sparse_attn_kernel(const __grid_constant__ CUtensorMap tmap_q, const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + OFF_Q;
    uint8_t* sKV = smem + OFF_KV;
    float* red = reinterpret_cast<float*>(smem + OFF_RED);
    float* m_neg = reinterpret_cast<float*>(smem + OFF_MNEG);
    float* alpha_s = reinterpret_cast<float*>(smem + OFF_ALPHA);
    float* invl_s = reinterpret_cast<float*>(smem + OFF_INVL);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* q_full = bars + 0;
    uint64_t* q_empty = bars + 1;
    uint64_t* seg_full = bars + 2;
    uint64_t* seg_free = bars + 7;   // latent chunk c (blocks 2c, 2c+1; chunk 3 also the rope block) consumed by PV
    uint64_t* s_full = bars + 7 + kSegs;
    uint64_t* p_full = s_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEM);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
    int* item_T = reinterpret_cast<int*>(smem + OFF_ITEM_T);

    const int warp = threadIdx.x / 32;
    const uint32_t lane = lane_id();

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, kIssuers);   // both issuers' last QK of an item read Q^T
        for (int c = 0; c < 5; ++c) mbar_init(&seg_full[c], kWorkers);  // one cp.async arrival per worker thread
        for (int c = 0; c < kSegs; ++c) mbar_init(&seg_free[c], 1);
        mbar_init(s_full, kIssuers);    // both partial sums of S^T
        mbar_init(p_full, kWorkerWarps);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmap_q);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    griddep_wait();                 // inputs and outputs may belong to the previous kernel until here

    if (warp == 0) {
        // ------------------------------------------------------------ Q loader (TMA)
        if (lane == 0) {
            int qi = 0;
            for (int s = 0;; ++s) {
                const int item = nth_item(p, s);
                if (item == -1) break;
                if (item < 0) continue;
                const Item I = decode_item(p, item);
                if (!mbar_wait_spin(q_empty, (qi & 1) ^ 1, abort_flag, p.status)) break;
                ++qi;
                mbar_arrive_expect_tx(q_full, 9 * kQBlkBytes);
                const int qrow = I.row * kH;
                for (int b = 0; b < 9; ++b) tma_load_2d(sQ + b * kQBlkBytes, &tmap_q, q_full, b * 64, qrow);
            }
        }
    } else if (warp <= kIssuers) {
        // ------------------------------------------------------------ MMA issuers
        // A single issuing thread keeps the tensor core at one M128 N64 K16 MMA per ~70 cycles;
        // two independent issuers reach one per ~48 (four are no faster).  The work splits by
        // 128-dim latent chunk: issuer 0 owns chunks 0 and 2, issuer 1 chunks 1 and 3 and the
        // rope block.  The owner of a chunk runs the QK over its dims into its own S^T partial
        // sum and the PV for that O^T chunk; the softmax adds the two partial sums.  The issuing
        // thread's instructions per MMA count: each descriptor is a precomputed base plus a
        // compile-time offset.
        const int iss = warp - 1;
        const uint32_t tm_s = tmem_base + TM_S + 64 * (uint32_t)iss;
        int gt = 0, qi = 0;
        bool ok = true;
        for (int s = 0; ok; ++s) {
            const int item = nth_item(p, s);
            if (item == -1) break;
            if (item < 0) continue;
            const Item I = decode_item(p, item);
            const int T = item_tiles(p, I, lane);
            if (lane == 0) {
                ok = mbar_wait_spin(q_full, qi & 1, abort_flag, p.status);
                const uint32_t kv_base = smem_u32(sKV);
                // operand descriptors at the buffers' starts; an MMA's descriptor is one of these
                // plus its operand's offset in 16-byte units (addresses stay below 256 KB, so the
                // 14-bit address field never carries)
                const uint64_t qk_a = sdesc_sw128(kv_base, 16, 1024);
                const uint64_t qk_b = sdesc_sw128(smem_u32(sQ), 16, 1024);
                // PV: A = V^T MN-major, 64-dim atoms 16 KB apart (LBO), 8-key groups 1 KB apart
                // (SBO); B = P^T MN-major, one 64-head atom, 8-key groups 1 KB apart
                const uint64_t pv_a = sdesc_sw128(kv_base, kBlkBytes, 1024);
                const uint64_t pv_b = sdesc_sw128(kv_base + 8 * kBlkBytes, kBlkBytes, 1024);
                bool q_released = false;
                for (int t = 0; ok && t < T; ++t, ++gt) {
                    // ---- this issuer's part of S^T = K . Q^T, segment by segment as the copies
                    // land: latent chunks iss and iss + 2, and for issuer 1 the rope block
                    // (segment 4).  Segment c's K blocks are 2c and 2c + 1 (the rope block is block
                    // 8), so its descriptors are the bases plus 2c blocks.  The accumulator needs
                    // no wait of its own: the previous tile's probabilities (p_full, awaited before
                    // its PV) were written after every worker had read both partial sums.
#pragma unroll
                    for (int j = 0; j < 3; ++j) {
                        if (j == 2 && iss == 0) break;
                        const int c = (j < 2) ? iss + 2 * j : 4;
                        if (!(ok = mbar_wait_spin(&seg_full[c], gt & 1, abort_flag, p.status))) break;
                        tc_fence_after();
                        const uint64_t a_c = qk_a + (uint64_t)(2 * c * (kBlkBytes >> 4));
                        const uint64_t b_c = qk_b + (uint64_t)(2 * c * (kQBlkBytes >> 4));
#pragma unroll
                        for (int bb = 0; bb < (j < 2 ? 2 : 1); ++bb) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_bf16_ss_lo(tm_s, (uint32_t)a_c + (uint32_t)(bb * (kBlkBytes >> 4) + 2 * kk),
                                               (uint32_t)(qk_a >> 32),
                                               (uint32_t)b_c + (uint32_t)(bb * (kQBlkBytes >> 4) + 2 * kk),
                                               (uint32_t)(qk_b >> 32), IDESC_QK, (j | bb | kk) ? 1u : 0u);
                        }
                    }
                    if (!ok) break;
                    mma_commit(s_full);
                    if (t == T - 1) {
                        mma_commit(q_empty);  // the next query's Q^T may stream in during the last softmax
                        q_released = true;
                    }
                    // ---- O^T += V^T . P^T for this issuer's 128-dim latent chunks: each
                    // chunk's blocks are freed as soon as it is consumed, so the next tile's
                    // copies of that chunk (and then its QK) overlap the rest of this PV
                    if (!(ok = mbar_wait_spin(p_full, gt & 1, abort_flag, p.status))) break;
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int c = iss + 2 * j;
                        const uint64_t a_c = pv_a + (uint64_t)(2 * c * (kBlkBytes >> 4));
                        const uint32_t d = tmem_base + TM_O + 64 * (uint32_t)c;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)   // 16 keys (two 8-key groups, 2 KB) per K step
                            mma_bf16_ss_lo(d, (uint32_t)a_c + (uint32_t)(kk * (2048 >> 4)), (uint32_t)(pv_a >> 32),
                                           (uint32_t)pv_b + (uint32_t)(kk * (2048 >> 4)), (uint32_t)(pv_b >> 32),
                                           IDESC_PV, (t > 0 || kk > 0) ? 1u : 0u);
                        // the copies of the rope block (which P^T overwrites) come after every
                        // chunk's free, so after every issuer's reads of P^T
                        mma_commit(&seg_free[c]);
                    }
                }
                if (ok && !q_released) mma_commit(q_empty);
                ++qi;
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
    } else {
        // ------------------------------------------------------------ workers (warps 3..18)
        const int ww = warp - 1 - kIssuers;       // 0..15
        const int quad = warp & 3;                // TMEM lane quadrant this warp may access
        const int hg = ww >> 2;                   // head group: heads h0 .. h0 + 15
        const int h0 = hg * kHG;
        // the head group's four warps (one per TMEM lane quadrant) agree on rescaling among themselves
        const uint32_t group_bar = 3 + (uint32_t)hg;
        const int tid = ww * 32 + (int)lane;      // 0..511
        const int key = quad * 32 + (int)lane;    // TMEM lane == key row of the tile == dim row of O^T
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        uint8_t* pT = sKV + 8 * kBlkBytes;
        const uint8_t* kv_bytes = reinterpret_cast<const uint8_t*>(p.kv);
        const uint32_t kv_smem = smem_u32(sKV);
        // PV of global tile g is complete once each issuer's last chunk (2 and 3) is free
        auto pv_done = [&](int g) -> bool {
            return worker_wait(&seg_free[kSegs - 2], g & 1, abort_flag, p.status) &&
                   worker_wait(&seg_free[kSegs - 1], g & 1, abort_flag, p.status);
        };

        // Gather cursor: walks this CTA's (item, tile) sequence one tile ahead
        // of the softmax.  Items without tiles are skipped here.  A worker warp
        // copies rows 64h + 4ww .. 64h + 4ww + 3 of each key half h.
        int g_s = 0, g_T = 0, g_t = 0, g_gt = 0;
        Item gI{};
        bool g_valid = false;
        int g_j = -1;  // lanes 0..7: key of row 64 (lane / 4) + 4 ww + lane % 4 of the cursor's tile
        // lanes 0..7: the key at the same row of the tile after the cursor's, with its batch and
        // bound; the next gather_issue prefetches that cache row into L2, one tile period before
        // its copy (a cache larger than what L2 keeps would otherwise put HBM latency on every
        // tile's critical path)
        int g_jn = -1, g_nbatch = 0, g_nbound = 0;
        auto g_advance_item = [&]() {
            g_valid = false;
            for (;;) {
                const int it = nth_item(p, g_s);
                if (it == -1) return;
                ++g_s;
                if (it < 0) continue;
                gI = decode_item(p, it);
                g_T = item_tiles(p, gI, lane);
                g_t = 0;
                if (g_T > 0) {
                    g_valid = true;
                    return;
                }
            }
        };
        // Load the cursor tile's row indices early, so that their latency hides
        // behind the softmax that precedes the copies.
        auto gather_prep = [&]() {
            g_j = -1;
            g_jn = -1;
            if (g_valid && lane < 8) {
                const int rowpos = 64 * (int)(lane >> 2) + 4 * ww + (int)(lane & 3);
                const int slot = gI.slot0 + g_t * kTile + rowpos;
                g_j = (slot < gI.slot_end) ? __ldg(p.idx + (int64_t)gI.row * p.top_k + slot) : -1;
                if (!PAGED && p.l2_prefetch) {
                    if (g_t + 1 < g_T) {
                        const int s2 = slot + kTile;
                        g_jn = (s2 < gI.slot_end) ? __ldg(p.idx + (int64_t)gI.row * p.top_k + s2) : -1;
                        g_nbatch = gI.batch;
                        g_nbound = gI.bound;
                    } else {
                        const int it = nth_item(p, g_s);   // the next item's first tile
                        if (it >= 0) {
                            const Item J = decode_item(p, it);
                            const int s2 = J.slot0 + rowpos;
                            g_jn = (s2 < J.slot_end) ? __ldg(p.idx + (int64_t)J.row * p.top_k + s2) : -1;
                            g_nbatch = J.batch;
                            g_nbound = J.bound;
                        }
                    }
                }
            }
        };
        // Issue this warp's copies of the cursor's tile, half by half as PV frees
        // them, then advance the cursor.  Returns false if a wait gave up.
        auto gather_issue = [&]() -> bool {
            if (!g_valid) return true;
            if (!PAGED && g_jn >= 0 && g_jn < g_nbound)   // g_jn stays -1 without l2_prefetch
                l2_prefetch_bulk(kv_bytes + ((int64_t)g_nbatch * p.Nmax + g_jn) * kRowBytes, kRowBytes);
            int j = g_j;
            if (j >= gI.bound) {
                raise_dev_error(p.status, DEV_ERR_BOUNDS);
                j = -1;
            }
            int64_t prow = (int64_t)gI.batch * p.Nmax + j;   // cache row of key j
            if (PAGED && j >= 0) {   // paged cache: the row's page from the sequence's table row
                const int page = __ldg(p.pages.table + (int64_t)gI.batch * p.pages.stride + (j >> p.pages.shift));
                if (page < 0 || page >= p.pages.num_pages) {
                    raise_dev_error(p.status, DEV_ERR_BOUNDS);
                    j = -1;
                } else {
                    prow = ((int64_t)page << p.pages.shift) + (j & ((1 << p.pages.shift) - 1));
                }
            }
            const uint8_t* src_row = (j >= 0) ? kv_bytes + prow * kRowBytes : kv_bytes;
            const uint32_t valid_mask = __ballot_sync(0xffffffffu, j >= 0);
            bool ok = true;
            // One warp instruction copies one 64-dim block (128 B) of four different rows, 8 lanes
            // per row: requests spread over many rows (and L2 slices) rather than long spans of one.
            // The warp's rows are 4 ww + i of each 64-key half h.
            const int i = (int)(lane >> 3);        // which of the warp's 4 rows of a half
            const int cc = lane & 7;               // 16-byte chunk of the 128-byte block
            const uint8_t* src_h[2];
            uint32_t nbytes_h[2], off_h[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = 64 * h + 4 * ww + i;
                src_h[h] = reinterpret_cast<const uint8_t*>(
                    __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(src_row), 4 * h + i)) + cc * 16;
                nbytes_h[h] = ((valid_mask >> (4 * h + i)) & 1u) ? 16u : 0u;
                off_h[h] = row * 128 + ((cc ^ (row & 7)) << 4);
            }
            for (int c = 0; c < kSegs; ++c) {
                ok = __all_sync(0xffffffffu, worker_wait(&seg_free[c], (g_gt & 1) ^ 1, abort_flag, p.status));
                if (!ok) break;
#pragma unroll
                for (int bb = 0; bb < 2; ++bb) {
                    const int blk = 2 * c + bb;
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        cp_async_16(kv_smem + blk * kBlkBytes + off_h[h], src_h[h] + blk * 128, nbytes_h[h]);
                }
                cp_async_arrive_noinc(&seg_full[c]);
                if (c == kSegs - 1) {   // the rope block: every chunk is free, so both issuers' reads of P^T are done
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        cp_async_16(kv_smem + 8 * kBlkBytes + off_h[h], src_h[h] + 8 * 128, nbytes_h[h]);
                    cp_async_arrive_noinc(&seg_full[4]);
                }
            }
            ++g_gt;
            if (++g_t >= g_T) g_advance_item();
            gather_prep();
            return ok;
        };

        // `gok` is this thread's wait status.  A wait that gives up (it also sets
        // the CTA's abort flag, so every later wait returns at once) does not
        // change the control flow inside an item: all workers keep meeting the
        // same named barriers, and the consensus barrier (bar.red.and over all
        // workers) at the end of the item takes every worker out together.
        g_advance_item();
        gather_prep();
        bool gok = gather_issue();
        bool failed = false;
        int gt = 0;
        for (int s = 0; !failed; ++s) {
            const int item = nth_item(p, s);
            if (item == -1) break;
            if (item < 0) continue;
            const Item I = decode_item(p, item);
            const int32_t* ir = p.idx + (int64_t)I.row * p.top_k;
            named_bar_sync(1, kWorkers);  // previous item's readers of m_neg / invl / item_T are done
            if (tid < kH) m_neg[tid] = kNoRef;
            if (ww == 0) {   // one warp finds the item's tile count for all
                const int tt = item_tiles(p, I, lane);
                if (lane == 0) *item_T = tt;
            }
            float2 l2[kHG / 2];   // row sums of heads (h0 + 2i, h0 + 2i + 1)
#pragma unroll
            for (int i = 0; i < kHG / 2; ++i) l2[i] = make_float2(0.f, 0.f);
            named_bar_sync(1, kWorkers);
            const int T = *item_T;
            for (int t = 0; t < T; ++t, ++gt) {
                const int slot = I.slot0 + t * kTile + key;
                const int j = (slot < I.slot_end) ? __ldg(ir + slot) : -1;  // issued before the wait
                gok = gok && worker_wait(s_full, gt & 1, abort_flag, p.status);
                tc_fence_after();
                const bool kvalid = (j >= 0) && (j < I.bound);
                // This key's scores for heads h0..h0+15 as pairs (packed f32x2 arithmetic): the two
                // issuers' partial sums added, plus -inf for a padding slot, so that neither the
                // reference check nor the probability needs the key's validity again.
                float2 x2[kHG / 2];
                {
                    uint32_t v[kHG], u[kHG];
                    tmem_ld16(tmem_base + lane_addr + TM_S + h0, v);
                    tmem_ld16(tmem_base + lane_addr + TM_S + 64 + h0, u);
                    tmem_ld_wait();
                    const float kb = kvalid ? 0.f : -INFINITY;
#pragma unroll
                    for (int i = 0; i < kHG / 2; ++i) {
                        const float2 a = make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                        const float2 b = make_float2(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
                        x2[i] = __fadd2_rn(__fadd2_rn(a, b), make_float2(kb, kb));
                    }
                }
                tc_fence_before();
                // Reference maxima (scaled, log2 units), one per head, kept negated: set from the
                // item's first tile, afterwards moved only when a score exceeds its head's reference
                // by more than 2^16 (checked per thread; rare), so the common path has no
                // cross-thread reduction.  The shifted exponent e = scale*log2(e)*s - m serves both
                // the check and the probability.  Before the first tile no reference is set (m_neg =
                // kNoRef), so any valid score counts as exceeding it, and a padding slot gives -inf,
                // which never does.  The scale is > 0, so maxima of the raw scores are maxima of the
                // scaled ones.
                const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
                float2 e2[kHG / 2];
#pragma unroll
                for (int h4 = 0; h4 < kHG / 4; ++h4) {
                    const float4 n4 = reinterpret_cast<const float4*>(m_neg + h0)[h4];
                    e2[2 * h4] = __ffma2_rn(x2[2 * h4], sc2, make_float2(n4.x, n4.y));
                    e2[2 * h4 + 1] = __ffma2_rn(x2[2 * h4 + 1], sc2, make_float2(n4.z, n4.w));
                }
                bool viol = false;
#pragma unroll
                for (int i = 0; i < kHG / 2; ++i) viol |= (e2[i].x > kRescaleThreshold) || (e2[i].y > kRescaleThreshold);
                const bool need_red = named_bar_or(group_bar, kGroupThreads, viol);
                bool any_upd = false;
                if (need_red) {
                    float xm[kHG];
#pragma unroll
                    for (int i = 0; i < kHG / 2; ++i) {
                        xm[2 * i] = x2[i].x;       // -inf for a padding slot
                        xm[2 * i + 1] = x2[i].y;
                    }
                    const float r = warp_transpose_reduce16<true>(xm, lane);
                    if ((lane & 1u) == 0) red[quad * kH + h0 + (int)(lane >> 1)] = r;
                    named_bar_sync(group_bar, kGroupThreads);
                    bool upd = false;
                    if (ww == 4 * hg && lane < kHG) {   // one lane per head of the group
                        const int h = h0 + (int)lane;
                        const float mt = p.scale_log2 * fmaxf(fmaxf(red[h], red[kH + h]), fmaxf(red[2 * kH + h], red[3 * kH + h]));
                        const bool unset = (m_neg[h] == kNoRef);
                        const float mo = -m_neg[h];
                        float a = 1.f;
                        if (mt > -INFINITY && (unset || mt > mo + kRescaleThreshold)) {
                            a = unset ? 0.f : ex2_approx(mo - mt);
                            m_neg[h] = -mt;
                            upd = !unset;
                        }
                        alpha_s[h] = a;
                    }
                    any_upd = named_bar_or(group_bar, kGroupThreads, upd);
#pragma unroll
                    for (int h4 = 0; h4 < kHG / 4; ++h4) {
                        const float4 n4 = reinterpret_cast<const float4*>(m_neg + h0)[h4];
                        e2[2 * h4] = __ffma2_rn(x2[2 * h4], sc2, make_float2(n4.x, n4.y));
                        e2[2 * h4 + 1] = __ffma2_rn(x2[2 * h4 + 1], sc2, make_float2(n4.z, n4.w));
                    }
                    if (any_upd) {
#pragma unroll
                        for (int h4 = 0; h4 < kHG / 4; ++h4) {
                            const float4 a4 = reinterpret_cast<const float4*>(alpha_s + h0)[h4];
                            l2[2 * h4] = __fmul2_rn(l2[2 * h4], make_float2(a4.x, a4.y));
                            l2[2 * h4 + 1] = __fmul2_rn(l2[2 * h4 + 1], make_float2(a4.z, a4.w));
                        }
                    }
                }
                // Probabilities: float32 into the row sum (so lse is the log of the exact sum),
                // rounded to bf16 for the MMA.
                uint32_t packed[kHG / 2];
#pragma unroll
                for (int i = 0; i < kHG / 2; ++i) {
                    const float2 pr = make_float2(ex2_approx(e2[i].x), ex2_approx(e2[i].y));
                    packed[i] = pack_bf16x2(pr.x, pr.y);
                    l2[i] = __fadd2_rn(l2[i], pr);
                }
                // P^T row `key`, heads h0..h0+15: 16-byte chunks 2hg and 2hg+1 of the swizzled 128-byte row
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int chunk = 2 * hg + i;
                    const uint4 v = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
                    *reinterpret_cast<uint4*>(pT + key * 128 + ((chunk ^ (key & 7)) << 4)) = v;
                }
                fence_proxy_async_smem();
                if (any_upd && t > 0) {
                    // O^T columns of the raised heads: wait for the previous PV (every chunk),
                    // then rescale in TMEM
                    gok = gok && pv_done(gt - 1);
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t v[kHG];
                        const uint32_t a = tmem_base + lane_addr + TM_O + 64 * c + h0;
                        tmem_ld16(a, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < kHG; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha_s[h0 + k]);
                        tmem_st16(a, v);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full);
                // copies of the next tile (this item's or the next item's first)
                gok = gather_issue() && gok;
            }
            // ---------------- final: l = sum of partial row sums; out = O^T / l
            {
                float l_part[kHG];
#pragma unroll
                for (int i = 0; i < kHG / 2; ++i) {
                    l_part[2 * i] = l2[i].x;
                    l_part[2 * i + 1] = l2[i].y;
                }
                const float r = warp_transpose_reduce16<false>(l_part, lane);
                if ((lane & 1u) == 0) red[quad * kH + h0 + (int)(lane >> 1)] = r;
            }
            if (!named_bar_and(2, kWorkers,
                               gok && (T == 0 || pv_done(gt - 1)))) {
                failed = true;
                break;
            }
            tc_fence_after();
            float lse_h = -INFINITY;
            if (tid < kH) {
                const float l = red[tid] + red[kH + tid] + red[2 * kH + tid] + red[3 * kH + tid];
                invl_s[tid] = (l > 0.f) ? 1.f / l : 0.f;
                lse_h = (l > 0.f) ? (log2f(l) - m_neg[tid]) * 0.6931471805599453f : -INFINITY;
            }
            named_bar_sync(1, kWorkers);
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                float o[kHG];
                if (T > 0) {
                    uint32_t v[kHG];
                    tmem_ld16(tmem_base + lane_addr + TM_O + 64 * c + h0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < kHG; ++h) o[h] = __uint_as_float(v[h]) * invl_s[h0 + h];
                } else {
#pragma unroll
                    for (int h = 0; h < kHG; ++h) o[h] = 0.f;
                }
                const int dim = c * 128 + key;
                if (PARTIAL) {
                    float* dst = p.part_o + (((int64_t)I.row * p.nsplit + I.split) * kH + h0) * kDv + dim;
#pragma unroll
                    for (int h = 0; h < kHG; ++h) dst[h * kDv] = o[h];
                } else if (p.out_f32) {
                    float* dst = static_cast<float*>(p.out) + ((int64_t)I.row * kH + h0) * kDv + dim;
#pragma unroll
                    for (int h = 0; h < kHG; ++h) dst[h * kDv] = o[h];
                } else {
                    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + ((int64_t)I.row * kH + h0) * kDv + dim;
#pragma unroll
                    for (int h = 0; h < kHG; ++h) dst[h * kDv] = __float2bfloat16_rn(o[h]);
                }
            }
            if (tid < kH) {
                if (PARTIAL)
                    p.part_lse[((int64_t)I.row * p.nsplit + I.split) * kH + tid] = lse_h;
                else if (p.lse)
                    p.lse[(int64_t)I.row * kH + tid] = lse_h;
            }
            tc_fence_before();
        }
        cp_async_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// Merge decode partials: out = sum_s exp(lse_s - M) o_s / sum_s exp(lse_s - M).
// A sequence has at most kMaxSplits splits (top_k <= DSA_MAX_TOPK, at least 128
// slots per split); every thread issues all of its split loads before using any.
constexpr int kMaxSplits = DSA_MAX_TOPK / kTile;
__global__ void __launch_bounds__(128) mla_decode_combine_kernel(const float* part_o, const float* part_lse,
                                                                 int nsplit, void* out, int out_f32, float* lse) {
    griddep_wait();
    const int b = blockIdx.x / kH, h = blockIdx.x % kH;
    const float* pl = part_lse + (int64_t)b * nsplit * kH + h;
    float ls[kMaxSplits];
    float4 v[kMaxSplits];
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) {
        ls[s] = (s < nsplit) ? pl[(int64_t)s * kH] : -INFINITY;
        v[s] = (s < nsplit) ? reinterpret_cast<const float4*>(part_o + (((int64_t)b * nsplit + s) * kH + h) * kDv)[threadIdx.x]
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) M = fmaxf(M, ls[s]);
    float wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) {
        const float wgt = (M == -INFINITY || ls[s] == -INFINITY) ? 0.f : expf(ls[s] - M);
        wsum += wgt;
        acc.x += wgt * v[s].x;
        acc.y += wgt * v[s].y;
        acc.z += wgt * v[s].z;
        acc.w += wgt * v[s].w;
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const int64_t o = ((int64_t)b * kH + h) * kDv + 4 * threadIdx.x;
    if (out_f32) {
        reinterpret_cast<float4*>(static_cast<float*>(out) + o)[0] =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(out) + o;
        dst[0] = __float2bfloat16_rn(acc.x * inv);
        dst[1] = __float2bfloat16_rn(acc.y * inv);
        dst[2] = __float2bfloat16_rn(acc.z * inv);
        dst[3] = __float2bfloat16_rn(acc.w * inv);
    }
    if (lse && threadIdx.x == 0) lse[(int64_t)b * kH + h] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

template <bool PARTIAL, bool PAGED>
dsa_status_t launch_kernel(const void* q, int q_rows, const AttnParams& prm, cudaStream_t stream) {
    CUtensorMap tq;
    dsa_status_t st = make_tmap_bf16_2d(&tq, q, kD, (uint64_t)q_rows * kH, kRowBytes, 64, kH);
    if (st != DSA_OK) return st;
    auto kern = mla_sparse_attn_kernel<PARTIAL, PAGED>;
    if ((st = ensure_smem_attr(reinterpret_cast<const void*>(kern), SMEM_BYTES)) != DSA_OK) return st;
    const int grid = min(prm.n_items, device_sm_count());
    if (launch_pdl(kern, dim3(grid), dim3(kThreads), SMEM_BYTES, stream, tq, prm) != cudaSuccess) return DSA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

// Splits per sequence for a decode launch: the B x splits items run on one persistent CTA per SM,
// so the launch takes about ceil(items / SMs) rounds of an item, and an item costs its tiles plus
// about two tiles' worth of fixed work (Q^T load, first-tile maxima, the partial's write and its
// share of the merge).  The split count with the least such cost wins, the smaller on a tie
// (fewer partials to merge).  Rounding the split count up from SMs / B instead left a second,
// mostly idle round at many batch sizes (B = 16: 160 items on 152 SMs).
int decode_splits(int B, int top_k) {
    const int tiles = ceil_div(top_k, kTile);
    const int sms = device_sm_count();
    int best = 1;
    long best_cost = -1;
    for (int ns = 1; ns <= tiles; ++ns) {
        const int per_item = ceil_div(tiles, ns);
        if (ns > 1 && ceil_div(tiles, ns - 1) == per_item) continue;   // same item length, more partials
        const long rounds = ceil_div(B * ns, sms);
        const long cost = rounds * (per_item + 2);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = ns;
        }
    }
    return best;
}

// Decode: prefetch the rows of an item's next tile into L2 when the caches the launch gathers from
// are large against L2 (see launch_attn_prefill) and an item has at least 8 tiles.  One persistent
// round of items leaves nothing to prefetch beyond an item's own tiles, and for 2-4 tile items the
// prefetches only compete with the copies (batch 16 / 32 at 4k keys: 27.3 -> 29.3 / 39.6 -> 41.6 us);
// at 16 tiles an item they gain 2-3% (batch 128 / 256).
int want_l2_prefetch_decode(size_t cache_bytes, int split_len) {
    return split_len >= 8 * kTile && cache_bytes > device_l2_bytes() / 4 ? 1 : 0;
}

}  // namespace

dsa_status_t launch_attn_prefill(const void* q, const void* kv, const int32_t* idx, int L, int N, int top_k,
                                 float scale, void* out, int out_f32, float* lse, const PageTable& pages,
                                 cudaStream_t stream) {
    AttnParams p{};
    p.kv = static_cast<const __nv_bfloat16*>(kv);
    p.idx = idx;
    p.kv_len = nullptr;
    p.out = out;
    p.out_f32 = out_f32;
    p.lse = lse;
    p.rows = L;
    p.prefill = 1;
    p.Nmax = N;
    p.top_k = top_k;
    p.nsplit = 1;
    p.split_len = ceil_div(top_k, kTile) * kTile;
    p.n_items = L;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.status = device_status_ptr();
    p.pages = pages;   // a paged cache: batch 0's table row
    // The gather reads each tile's rows at random from the cache; once the cache is large against
    // L2 (measured: a 75 MB cache at a 59% L2 hit rate, a 19 MB one at 94%), each tile's copies
    // wait for HBM unless their rows were prefetched.  For an L2-resident cache the prefetches
    // only cost issue slots (1.8% at 19 MB), so they are enabled above a quarter of L2.
    p.l2_prefetch = (size_t)N * kRowBytes > device_l2_bytes() / 4 ? 1 : 0;
    return p.pages.table ? launch_kernel<false, true>(q, L, p, stream) : launch_kernel<false, false>(q, L, p, stream);
}

size_t attn_decode_workspace(int B, int top_k) {
    const int ns = ceil_div(top_k, kTile);  // upper bound on the splits the launcher may pick
    return (size_t)B * ns * kH * (kDv + 1) * sizeof(float) + 256;
}

dsa_status_t launch_attn_decode(const void* q, const void* kv, const int32_t* kv_len, const int32_t* idx, int B,
                                int Nmax, int top_k, float scale, void* out, int out_f32, float* lse,
                                void* workspace, const PageTable& pages, cudaStream_t stream) {
    const int ns = decode_splits(B, top_k);
    const int tiles = ceil_div(top_k, kTile);
    AttnParams p{};
    p.kv = static_cast<const __nv_bfloat16*>(kv);
    p.idx = idx;
    p.kv_len = kv_len;
    p.part_o = static_cast<float*>(workspace);
    p.part_lse = p.part_o + (size_t)B * ns * kH * kDv;
    p.rows = B;
    p.prefill = 0;
    p.Nmax = Nmax;
    p.top_k = top_k;
    p.nsplit = ns;
    p.split_len = ceil_div(tiles, ns) * kTile;
    p.nsplit = ceil_div(top_k, p.split_len);
    p.n_items = B * p.nsplit;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.status = device_status_ptr();
    p.pages = pages;
    p.l2_prefetch = want_l2_prefetch_decode((size_t)B * Nmax * kRowBytes, p.split_len);
    dsa_status_t st = p.pages.table ? launch_kernel<true, true>(q, B, p, stream) : launch_kernel<true, false>(q, B, p, stream);
    if (st != DSA_OK) return st;
    if (launch_pdl(mla_decode_combine_kernel, dim3(B * kH), dim3(128), 0, stream, (const float*)p.part_o,
                   (const float*)p.part_lse, p.nsplit, out, out_f32, lse) != cudaSuccess)
        return DSA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Allocation-free decode (mla_sparse_attn_decode_noalloc).  For callers that
// may not allocate device memory, the split partials live in this fixed
// file-scope array instead of a caller workspace.  Its name is only a host-side
// stand-in for the device object, so the host looks up the real device address
// once per device (cudaGetSymbolAddress, no allocation) and passes it to the
// kernels.  All calls on a device share it; overlapping calls race.
namespace {
constexpr size_t kNoallocScratchBytes = DSA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevicesNoalloc = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevicesNoalloc] = {};

dsa_status_t noalloc_scratch(void** ptr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return DSA_ERR_CUDA;
    if (dev >= kMaxDevicesNoalloc) return DSA_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> g(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, g_noalloc_scratch) != cudaSuccess || !a) return DSA_ERR_CUDA;
        g_noalloc_ptr[dev] = a;
    }
    *ptr = g_noalloc_ptr[dev];
    return DSA_OK;
}
}  // namespace

dsa_status_t launch_attn_decode_noalloc(const void* q, const void* kv, const int32_t* kv_len, const int32_t* idx,
                                        int B, int Nmax, int top_k, float scale, void* out, int out_f32,
                                        float* lse, cudaStream_t stream) {
    const size_t per_item = (size_t)kH * (kDv + 1) * sizeof(float);
    const int max_items = (int)(kNoallocScratchBytes / per_item);
    if (B > max_items) return DSA_ERR_SCRATCH_TOO_SMALL;
    void* scratch = nullptr;
    dsa_status_t st = noalloc_scratch(&scratch);
    if (st != DSA_OK) return st;
    const int tiles = ceil_div(top_k, kTile);
    int ns = decode_splits(B, top_k);
    if (ns > max_items / B) ns = max_items / B;
    if (ns < 1) ns = 1;
    AttnParams p{};
    p.kv = static_cast<const __nv_bfloat16*>(kv);
    p.idx = idx;
    p.kv_len = kv_len;
    p.part_o = static_cast<float*>(scratch);
    p.rows = B;
    p.prefill = 0;
    p.Nmax = Nmax;
    p.top_k = top_k;
    p.split_len = ceil_div(tiles, ns) * kTile;
    p.nsplit = ceil_div(top_k, p.split_len);
    p.part_lse = p.part_o + (size_t)B * p.nsplit * kH * kDv;
    p.n_items = B * p.nsplit;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.status = device_status_ptr();
    p.l2_prefetch = want_l2_prefetch_decode((size_t)B * Nmax * kRowBytes, p.split_len);
    st = launch_kernel<true, false>(q, B, p, stream);
    if (st != DSA_OK) return st;
    if (launch_pdl(mla_decode_combine_kernel, dim3(B * kH), dim3(128), 0, stream, (const float*)p.part_o,
                   (const float*)p.part_lse, p.nsplit, out, out_f32, lse) != cudaSuccess)
        return DSA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
