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
//   * Gather: 4 warps issue 16-byte cp.async copies of the selected rows,
//     straight into the swizzled layout, in 5 segments (4 latent 128-dim
//     chunks + the rope block).  Each segment has its own full/free barrier so
//     the next tile's chunk c streams in as soon as PV has consumed chunk c.
//     Unselected or padding slots are zero-filled (never NaN garbage).
//   * Softmax: 4 warps, one key per thread.  Each head's reference maximum is
//     taken from the query's first tile (transposing warp butterfly + one
//     shared-memory exchange); later tiles only check, per thread, whether a
//     score exceeds its reference by more than 2^16, and only then reduce and
//     rescale O^T in TMEM.  Numerator and denominator always share the
//     reference, so the result is the exact softmax.  P^T is written as bf16
//     into the (consumed) rope block.
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
constexpr int kThreads = 320;          // 10 warps
constexpr float kRescaleThreshold = 16.0f;  // log2 units

// smem layout (1024-aligned base)
constexpr int OFF_Q = 0;                               // 9 x 8 KB
constexpr int OFF_KV = OFF_Q + 9 * kQBlkBytes;         // 9 x 16 KB (block 8 = rope, then P^T)
constexpr int OFF_RED = OFF_KV + 9 * kBlkBytes;        // float [4][64]
constexpr int OFF_MUSED = OFF_RED + 4 * kH * 4;        // float [64]
constexpr int OFF_ALPHA = OFF_MUSED + kH * 4;          // float [64]
constexpr int OFF_INVL = OFF_ALPHA + kH * 4;           // float [64]
constexpr int OFF_BAR = OFF_INVL + kH * 4;
// barriers: q_full, q_empty, seg_full[5], seg_free[5], s_full, s_empty, p_full, pv_done
constexpr int N_BARS = 2 + 5 + 5 + 4;
constexpr int OFF_TMEM = OFF_BAR + N_BARS * 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int SMEM_BYTES = OFF_ABORT + 4 + 1024;

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;      // S^T: 64 columns
constexpr uint32_t TM_O = 64;     // O^T chunk c at 64 + 64 c

constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 64, true, true);

struct AttnParams {
    const __nv_bfloat16* kv;   // [B][Nmax][576]
    const int32_t* idx;        // [rows][top_k]
    const int32_t* kv_len;     // [B] or nullptr (then every row may use Nmax keys)
    __nv_bfloat16* out;        // final: [rows][64][512]
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
};

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
// slot range (warp-collective; every lane gets the same answer).
__device__ __forceinline__ int item_tiles(const AttnParams& p, const Item& I, uint32_t lane) {
    const int32_t* ir = p.idx + (int64_t)I.row * p.top_k;
    for (int base = I.slot_end - 32; base > I.slot0 - 32; base -= 32) {
        const int s = base + (int)lane;
        const bool v = (s >= I.slot0) && (s < I.slot_end) && (__ldg(ir + s) >= 0);
        const uint32_t m = __ballot_sync(0xffffffffu, v);
        if (m) {
            const int last = base + 31 - __clz(m);
            return (last - I.slot0) / kTile + 1;
        }
    }
    return 0;
}

// Transposing butterfly over a warp: on entry every lane holds 64 values (one
// per head); on exit lane l holds the warp-wide reduction for heads 2l, 2l+1.
template <bool MAX>
__device__ __forceinline__ void warp_transpose_reduce(const float (&x)[64], uint32_t lane, float& r0, float& r1) {
    float a[32];
    {
        const bool up = lane & 16;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            float mine = up ? x[32 + k] : x[k];
            float other = up ? x[k] : x[32 + k];
            float recv = __shfl_xor_sync(0xffffffffu, other, 16);
            a[k] = MAX ? fmaxf(mine, recv) : mine + recv;
        }
    }
#pragma unroll
    for (int step = 0; step < 4; ++step) {
        const int half = 16 >> step;         // 16, 8, 4, 2 values kept
        const int off = 8 >> step;           // shuffle distance 8, 4, 2, 1
        const bool up = lane & off;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (k < half) {
                float mine = up ? a[half + k] : a[k];
                float other = up ? a[k] : a[half + k];
                float recv = __shfl_xor_sync(0xffffffffu, other, off);
                a[k] = MAX ? fmaxf(mine, recv) : mine + recv;
            }
        }
    }
    r0 = a[0];
    r1 = a[1];
}

template <bool PARTIAL>
__global__ void __launch_bounds__(kThreads, 1)
    mla_sparse_attn_kernel(const __grid_constant__ CUtensorMap tmap_q, const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + OFF_Q;
    uint8_t* sKV = smem + OFF_KV;
    float* red = reinterpret_cast<float*>(smem + OFF_RED);
    float* m_used = reinterpret_cast<float*>(smem + OFF_MUSED);
    float* alpha_s = reinterpret_cast<float*>(smem + OFF_ALPHA);
    float* invl_s = reinterpret_cast<float*>(smem + OFF_INVL);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* q_full = bars + 0;
    uint64_t* q_empty = bars + 1;
    uint64_t* seg_full = bars + 2;
    uint64_t* seg_free = bars + 7;
    uint64_t* s_full = bars + 12;
    uint64_t* s_empty = bars + 13;
    uint64_t* p_full = bars + 14;
    uint64_t* pv_done = bars + 15;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEM);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);

    const int warp = threadIdx.x / 32;
    const uint32_t lane = lane_id();

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int c = 0; c < 5; ++c) {
            mbar_init(&seg_full[c], 128);
            mbar_init(&seg_free[c], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_empty, 128);
        mbar_init(p_full, 128);
        mbar_init(pv_done, 1);
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

    if (warp == 0) {
        // ------------------------------------------------------------ Q loader (TMA)
        if (lane == 0) {
            int qi = 0;
            for (int s = 0;; ++s) {
                const int item = nth_item(p, s);
                if (item == -1) break;
                if (item < 0) continue;
                const Item I = decode_item(p, item);
                if (!mbar_wait(q_empty, (qi & 1) ^ 1, abort_flag, p.status)) break;
                ++qi;
                mbar_arrive_expect_tx(q_full, 9 * kQBlkBytes);
                const int qrow = I.row * kH;
                for (int b = 0; b < 9; ++b) tma_load_2d(sQ + b * kQBlkBytes, &tmap_q, q_full, b * 64, qrow);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        int gt = 0, qi = 0;
        bool ok = true;
        for (int s = 0; ok; ++s) {
            const int item = nth_item(p, s);
            if (item == -1) break;
            if (item < 0) continue;
            const Item I = decode_item(p, item);
            const int T = item_tiles(p, I, lane);
            if (lane == 0) {
                ok = mbar_wait(q_full, qi & 1, abort_flag, p.status);
                const uint32_t q_base = smem_u32(sQ);
                const uint32_t kv_base = smem_u32(sKV);
                for (int t = 0; ok && t < T; ++t, ++gt) {
                    // ---- S^T = K . Q^T over the 576 dims, segment by segment
                    if (!(ok = mbar_wait(s_empty, (gt & 1) ^ 1, abort_flag, p.status))) break;
                    for (int c = 0; c < 5 && ok; ++c) {
                        if (!(ok = mbar_wait(&seg_full[c], gt & 1, abort_flag, p.status))) break;
                        tc_fence_after();
                        const int b_lo = (c < 4) ? 2 * c : 8;
                        const int nb = (c < 4) ? 2 : 1;
                        for (int bb = 0; bb < nb; ++bb) {
                            const int blk = b_lo + bb;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint64_t ad = sdesc_sw128(kv_base + blk * kBlkBytes + kk * 32, 16, 1024);
                                const uint64_t bd = sdesc_sw128(q_base + blk * kQBlkBytes + kk * 32, 16, 1024);
                                mma_bf16_ss(tmem_base + TM_S, ad, bd, IDESC_QK, (c | bb | kk) != 0);
                            }
                        }
                    }
                    if (!ok) break;
                    mma_commit(s_full);
                    // ---- O^T += V^T . P^T, 128 latent dims per chunk
                    if (!(ok = mbar_wait(p_full, gt & 1, abort_flag, p.status))) break;
                    tc_fence_after();
                    const uint32_t p_base = kv_base + 8 * kBlkBytes;
                    for (int c = 0; c < 4; ++c) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            // A = V^T: MN-major, 64-dim atoms 16 KB apart (LBO), 8-key groups 1 KB apart (SBO)
                            const uint64_t ad =
                                sdesc_sw128(kv_base + (2 * c) * kBlkBytes + kk * 2048, kBlkBytes, 1024);
                            // B = P^T: MN-major, one 64-head atom, 8-key groups 1 KB apart
                            const uint64_t bd = sdesc_sw128(p_base + kk * 2048, kBlkBytes, 1024);
                            mma_bf16_ss(tmem_base + TM_O + 64 * c, ad, bd, IDESC_PV, (t > 0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(&seg_free[c]);
                    }
                    mma_commit(&seg_free[4]);
                    mma_commit(pv_done);
                }
                if (ok) mma_commit(q_empty);
                ++qi;
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ gather (warps 2..5)
        const int gw = warp - 2;
        const uint8_t* kv_bytes = reinterpret_cast<const uint8_t*>(p.kv);
        int gt = 0;
        bool ok = true;
        for (int s = 0; ok; ++s) {
            const int item = nth_item(p, s);
            if (item == -1) break;
            if (item < 0) continue;
            const Item I = decode_item(p, item);
            const int T = item_tiles(p, I, lane);
            const int32_t* ir = p.idx + (int64_t)I.row * p.top_k;
            const uint8_t* kv_batch = kv_bytes + (int64_t)I.batch * p.Nmax * kRowBytes;
            for (int t = 0; t < T; ++t, ++gt) {
                // this lane's row of the tile: gw*32 + lane
                const int slot = I.slot0 + t * kTile + gw * 32 + (int)lane;
                int j = (slot < I.slot_end) ? __ldg(ir + slot) : -1;
                if (j >= I.bound) {
                    raise_dev_error(p.status, DEV_ERR_BOUNDS);
                    j = -1;
                }
                const uint8_t* src_row = (j >= 0) ? kv_batch + (int64_t)j * kRowBytes : kv_bytes;
                const uint32_t valid_mask = __ballot_sync(0xffffffffu, j >= 0);
                for (int c = 0; c < 5; ++c) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&seg_free[c], (gt & 1) ^ 1, abort_flag, p.status));
                    if (!ok) break;
                    if (c < 4) {
                        // 128 dims = 16 chunks of 16 B per row; two rows per warp instruction
                        const int chunk = lane & 15;
                        const int blk = 2 * c + (chunk >> 3);
                        const int cc = chunk & 7;
#pragma unroll 4
                        for (int s2 = 0; s2 < 16; ++s2) {
                            const int rl = 2 * s2 + (int)(lane >> 4);   // row within this warp's 32
                            const int row = gw * 32 + rl;
                            const uint8_t* src = reinterpret_cast<const uint8_t*>(
                                __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(src_row), rl));
                            const bool v = (valid_mask >> rl) & 1u;
                            const uint32_t dst =
                                smem_u32(sKV) + blk * kBlkBytes + row * 128 + ((cc ^ (row & 7)) << 4);
                            cp_async_16(dst, src + (c * 16 + chunk) * 16, v ? 16u : 0u);
                        }
                    } else {
                        // rope: 64 dims = 8 chunks per row; four rows per warp instruction
                        const int cc = lane & 7;
#pragma unroll 4
                        for (int s2 = 0; s2 < 8; ++s2) {
                            const int rl = 4 * s2 + (int)(lane >> 3);
                            const int row = gw * 32 + rl;
                            const uint8_t* src = reinterpret_cast<const uint8_t*>(
                                __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(src_row), rl));
                            const bool v = (valid_mask >> rl) & 1u;
                            const uint32_t dst =
                                smem_u32(sKV) + 8 * kBlkBytes + row * 128 + ((cc ^ (row & 7)) << 4);
                            cp_async_16(dst, src + (64 + cc) * 16, v ? 16u : 0u);
                        }
                    }
                    cp_async_arrive_noinc(&seg_full[c]);
                }
                if (!ok) break;
            }
        }
        cp_async_wait_all();
    } else {
        // ------------------------------------------------------------ softmax + epilogue (warps 6..9)
        const int sw = warp - 6;                 // 0..3
        const int quad = warp & 3;               // TMEM lane quadrant
        const int tid = sw * 32 + (int)lane;     // 0..127
        const int key = quad * 32 + (int)lane;   // TMEM lane == key row of the tile == dim row of O^T
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        uint8_t* pT = sKV + 8 * kBlkBytes;
        int gt = 0;
        bool ok = true;
        for (int s = 0; ok; ++s) {
            const int item = nth_item(p, s);
            if (item == -1) break;
            if (item < 0) continue;
            const Item I = decode_item(p, item);
            const int T = item_tiles(p, I, lane);
            const int32_t* ir = p.idx + (int64_t)I.row * p.top_k;
            named_bar_sync(1, 128);  // previous item's readers of m_used / invl are done
            if (tid < kH) m_used[tid] = -INFINITY;
            float l_part[kH];
#pragma unroll
            for (int h = 0; h < kH; ++h) l_part[h] = 0.f;
            named_bar_sync(1, 128);
            for (int t = 0; t < T; ++t, ++gt) {
                ok = named_bar_and(2, 128, mbar_wait(s_full, gt & 1, abort_flag, p.status));
                if (!ok) break;
                tc_fence_after();
                float x[kH];
                {
                    uint32_t v0[32], v1[32];
                    tmem_ld32(tmem_base + lane_addr + TM_S, v0);
                    tmem_ld32(tmem_base + lane_addr + TM_S + 32, v1);
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < 32; ++h) {
                        x[h] = __uint_as_float(v0[h]);
                        x[32 + h] = __uint_as_float(v1[h]);
                    }
                }
                tc_fence_before();
                mbar_arrive(s_empty);
                const int slot = I.slot0 + t * kTile + key;
                int j = (slot < I.slot_end) ? __ldg(ir + slot) : -1;
                if (!((j >= 0) && (j < I.bound))) {
#pragma unroll
                    for (int h = 0; h < kH; ++h) x[h] = -INFINITY;
                }
                // Reference maxima (scaled, log2 units): set from the item's first tile.
                // Afterwards a head's reference only moves when one of its scores exceeds
                // it by more than 2^16 (checked per thread; rare), so the common path has
                // no cross-thread reduction.  The scale is > 0, so maxima of the raw
                // scores are maxima of the scaled ones.
                bool need_red = (t == 0);
                if (!need_red) {
                    bool viol = false;
#pragma unroll
                    for (int h4 = 0; h4 < kH / 4; ++h4) {
                        const float4 m4 = reinterpret_cast<const float4*>(m_used)[h4];
                        viol |= x[4 * h4 + 0] * p.scale_log2 > m4.x + kRescaleThreshold;
                        viol |= x[4 * h4 + 1] * p.scale_log2 > m4.y + kRescaleThreshold;
                        viol |= x[4 * h4 + 2] * p.scale_log2 > m4.z + kRescaleThreshold;
                        viol |= x[4 * h4 + 3] * p.scale_log2 > m4.w + kRescaleThreshold;
                    }
                    need_red = named_bar_or(1, 128, viol);
                }
                bool any_upd = false;
                if (need_red) {
                    float r0, r1;
                    warp_transpose_reduce<true>(x, lane, r0, r1);
                    red[sw * kH + 2 * lane] = r0;
                    red[sw * kH + 2 * lane + 1] = r1;
                    named_bar_sync(1, 128);
                    bool upd = false;
                    if (tid < kH) {
                        const float mt = p.scale_log2 * fmaxf(fmaxf(red[tid], red[kH + tid]),
                                                              fmaxf(red[2 * kH + tid], red[3 * kH + tid]));
                        const float mo = m_used[tid];
                        float a = 1.f;
                        if (mt > -INFINITY && (mo == -INFINITY || mt > mo + kRescaleThreshold)) {
                            a = (mo == -INFINITY) ? 0.f : ex2_approx(mo - mt);
                            m_used[tid] = mt;
                            upd = (mo != -INFINITY);
                        }
                        alpha_s[tid] = a;
                    }
                    any_upd = named_bar_or(1, 128, upd);
                }
                // probabilities (bf16 for the MMA, float32 for the row sum)
                uint32_t packed[kH / 2];
#pragma unroll
                for (int h4 = 0; h4 < kH / 4; ++h4) {
                    const float4 m4 = reinterpret_cast<const float4*>(m_used)[h4];
                    const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
                    float pr[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        pr[k] = ex2_approx(fmaf(x[4 * h4 + k], p.scale_log2, (mm[k] == -INFINITY) ? 0.f : -mm[k]));
                    if (any_upd) {
                        const float4 a4 = reinterpret_cast<const float4*>(alpha_s)[h4];
                        l_part[4 * h4 + 0] *= a4.x;
                        l_part[4 * h4 + 1] *= a4.y;
                        l_part[4 * h4 + 2] *= a4.z;
                        l_part[4 * h4 + 3] *= a4.w;
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) l_part[4 * h4 + k] += pr[k];
                    packed[2 * h4] = pack_bf16x2(pr[0], pr[1]);
                    packed[2 * h4 + 1] = pack_bf16x2(pr[2], pr[3]);
                }
                // P^T row `key`: 64 heads x bf16 = 128 B, 128-byte swizzle
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    uint4 v = make_uint4(packed[4 * cc], packed[4 * cc + 1], packed[4 * cc + 2], packed[4 * cc + 3]);
                    *reinterpret_cast<uint4*>(pT + key * 128 + ((cc ^ (key & 7)) << 4)) = v;
                }
                fence_proxy_async_smem();
                if (any_upd && t > 0) {
                    // O^T columns of the raised heads: wait for the previous PV, then rescale in TMEM
                    ok = named_bar_and(2, 128, mbar_wait(pv_done, (gt - 1) & 1, abort_flag, p.status));
                    if (!ok) break;
                    tc_fence_after();
                    for (int c = 0; c < 4; ++c) {
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            uint32_t v[32];
                            const uint32_t a = tmem_base + lane_addr + TM_O + 64 * c + 32 * hh;
                            tmem_ld32(a, v);
                            tmem_ld_wait();
#pragma unroll
                            for (int k = 0; k < 32; ++k)
                                v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha_s[32 * hh + k]);
                            tmem_st32(a, v);
                        }
                    }
                    tmem_st_wait();
                    tc_fence_before();
                }
                mbar_arrive(p_full);
            }
            if (!ok) break;
            // ---------------- final: l = sum of partial row sums; out = O^T / l
            float r0, r1;
            warp_transpose_reduce<false>(l_part, lane, r0, r1);
            red[sw * kH + 2 * lane] = r0;
            red[sw * kH + 2 * lane + 1] = r1;
            if (T > 0) {
                ok = named_bar_and(2, 128, mbar_wait(pv_done, (gt - 1) & 1, abort_flag, p.status));
                if (!ok) break;
                tc_fence_after();
            } else {
                named_bar_sync(1, 128);
            }
            float lse_h = -INFINITY;
            if (tid < kH) {
                const float l = red[tid] + red[kH + tid] + red[2 * kH + tid] + red[3 * kH + tid];
                invl_s[tid] = (l > 0.f) ? 1.f / l : 0.f;
                lse_h = (l > 0.f) ? (m_used[tid] + log2f(l)) * 0.6931471805599453f : -INFINITY;
            }
            named_bar_sync(1, 128);
            for (int c = 0; c < 4; ++c) {
                float o[kH];
                if (T > 0) {
                    uint32_t v0[32], v1[32];
                    tmem_ld32(tmem_base + lane_addr + TM_O + 64 * c, v0);
                    tmem_ld32(tmem_base + lane_addr + TM_O + 64 * c + 32, v1);
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < 32; ++h) {
                        o[h] = __uint_as_float(v0[h]) * invl_s[h];
                        o[32 + h] = __uint_as_float(v1[h]) * invl_s[32 + h];
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < kH; ++h) o[h] = 0.f;
                }
                const int dim = c * 128 + key;
                if (PARTIAL) {
                    float* dst = p.part_o + ((int64_t)I.row * p.nsplit + I.split) * kH * kDv + dim;
#pragma unroll
                    for (int h = 0; h < kH; ++h) dst[h * kDv] = o[h];
                } else {
                    __nv_bfloat16* dst = p.out + (int64_t)I.row * kH * kDv + dim;
#pragma unroll
                    for (int h = 0; h < kH; ++h) dst[h * kDv] = __float2bfloat16_rn(o[h]);
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
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// Merge decode partials: out = sum_s exp(lse_s - M) o_s / sum_s exp(lse_s - M).
__global__ void __launch_bounds__(128) mla_decode_combine_kernel(const float* part_o, const float* part_lse,
                                                                 int nsplit, __nv_bfloat16* out, float* lse) {
    const int b = blockIdx.x / kH, h = blockIdx.x % kH;
    const float* pl = part_lse + (int64_t)b * nsplit * kH + h;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, pl[(int64_t)s * kH]);
    float wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < nsplit; ++s) {
        const float ls = pl[(int64_t)s * kH];
        const float wgt = (M == -INFINITY) ? 0.f : expf(ls - M);
        wsum += wgt;
        const float4 v = reinterpret_cast<const float4*>(part_o + (((int64_t)b * nsplit + s) * kH + h) * kDv)[threadIdx.x];
        acc.x += wgt * v.x;
        acc.y += wgt * v.y;
        acc.z += wgt * v.z;
        acc.w += wgt * v.w;
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    __nv_bfloat16* dst = out + ((int64_t)b * kH + h) * kDv + 4 * threadIdx.x;
    dst[0] = __float2bfloat16_rn(acc.x * inv);
    dst[1] = __float2bfloat16_rn(acc.y * inv);
    dst[2] = __float2bfloat16_rn(acc.z * inv);
    dst[3] = __float2bfloat16_rn(acc.w * inv);
    if (lse && threadIdx.x == 0) lse[(int64_t)b * kH + h] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

template <bool PARTIAL>
dsa_status_t launch_kernel(const void* q, int q_rows, const AttnParams& prm, cudaStream_t stream) {
    CUtensorMap tq;
    dsa_status_t st = make_tmap_bf16_2d(&tq, q, kD, (uint64_t)q_rows * kH, kRowBytes, 64, kH);
    if (st != DSA_OK) return st;
    auto kern = mla_sparse_attn_kernel<PARTIAL>;
    if ((st = ensure_smem_attr(reinterpret_cast<const void*>(kern), SMEM_BYTES)) != DSA_OK) return st;
    const int grid = min(prm.n_items, device_sm_count());
    kern<<<grid, kThreads, SMEM_BYTES, stream>>>(tq, prm);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int decode_splits(int B, int top_k) {
    const int tiles = ceil_div(top_k, kTile);
    int ns = ceil_div(device_sm_count(), B);
    if (ns > tiles) ns = tiles;
    if (ns < 1) ns = 1;
    return ns;
}

}  // namespace

dsa_status_t launch_attn_prefill(const void* q, const void* kv, const int32_t* idx, int L, int N, int top_k,
                                 float scale, void* out, float* lse, cudaStream_t stream) {
    AttnParams p{};
    p.kv = static_cast<const __nv_bfloat16*>(kv);
    p.idx = idx;
    p.kv_len = nullptr;
    p.out = static_cast<__nv_bfloat16*>(out);
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
    return launch_kernel<false>(q, L, p, stream);
}

size_t attn_decode_workspace(int B, int top_k) {
    const int ns = ceil_div(top_k, kTile);  // upper bound on the splits the launcher may pick
    return (size_t)B * ns * kH * (kDv + 1) * sizeof(float) + 256;
}

dsa_status_t launch_attn_decode(const void* q, const void* kv, const int32_t* kv_len, const int32_t* idx, int B,
                                int Nmax, int top_k, float scale, void* out, float* lse, void* workspace,
                                cudaStream_t stream) {
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
    dsa_status_t st = launch_kernel<true>(q, B, p, stream);
    if (st != DSA_OK) return st;
    mla_decode_combine_kernel<<<B * kH, 128, 0, stream>>>(p.part_o, p.part_lse, p.nsplit,
                                                         static_cast<__nv_bfloat16*>(out), lse);
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
                                        int B, int Nmax, int top_k, float scale, void* out, float* lse,
                                        cudaStream_t stream) {
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
    st = launch_kernel<true>(q, B, p, stream);
    if (st != DSA_OK) return st;
    mla_decode_combine_kernel<<<B * kH, 128, 0, stream>>>(p.part_o, p.part_lse, p.nsplit,
                                                         static_cast<__nv_bfloat16*>(out), lse);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
