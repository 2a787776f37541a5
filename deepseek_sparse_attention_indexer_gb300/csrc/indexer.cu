// indexer.cu -- DSA indexer scores on the sm_103a tensor cores.
//
// What it computes (exo PR #2539, GLM-5.2/5.3 attention, section "Prefill",
// bullet "Indexer scores in float32, in one kernel"): for every causal
// (query i, key j), S[i,j] = sum over the 32 indexer heads h of
// w[i,h] * relu(qI[i,h,:] . kI[j,:]), summed in float32 in one pass, with the
// causal mask applied (masked keys hold -inf).
//
// How (GB300 design):
//   * One tcgen05 MMA per key tile: M = 128 keys (the A operand, streamed by
//     TMA through a 4-stage ring), N = 4 queries x 32 heads = 128 (the B
//     operand, the group's indexer queries, resident while the CTA walks its
//     key range), K = 128 (head dim).  The accumulator D[key, (q,h)] lands in
//     TMEM, four deep (4 x 128 columns), so the MMAs run up to three tiles
//     ahead of the epilogue.
//   * Because the keys sit on the TMEM lanes, the 32-head reduction of one
//     (query, key) score lives entirely inside one thread: 32 columns of its
//     lane, relu, times the head weight, summed -- no cross-thread traffic and
//     no per-head [L, N] tensor ever exists.  Each warp then stores 32
//     consecutive keys of a score row (128-byte coalesced stores).
//   * Warp roles: warp 0 issues TMA, warps 1 and 2 issue the MMAs (one thread
//     each, alternating key tiles), warps 3..18 run the epilogue, four per TMEM
//     lane quadrant, one query each:
//     with four epilogue warps per scheduler, one warp's TMEM loads hide
//     behind the others' arithmetic, and a warp's query keeps its 32 head
//     weights in registers for the whole item.  (Eight-query groups, N = 256,
//     read each key tile half as often but give a warp two queries, whose 64
//     weights do not fit in 96 registers: re-reading them, as broadcast loads,
//     on every tile made those groups 18-22% slower on GB300.)
//   * Work items are (batch, 4-query group, key chunk); CTAs are persistent and
//     walk the items in a zig-zag order so the triangular causal workload of a
//     first chunk spreads evenly.  Key tiles past the group's last causal key
//     issue no MMA: the epilogue only writes -inf there.
//   * Decode (one query per sequence) uses the same kernel with N = 32.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {

namespace {

constexpr int kHi = DSA_INDEXER_HEADS;  // 32
constexpr int kDi = DSA_INDEXER_DIM;    // 128
constexpr int kTileKeys = 128;          // MMA M
constexpr int kEpiWarps = 16;           // four per TMEM lane quadrant, one query each
constexpr int kIssuers = 2;              // MMA-issuing warps, alternating key tiles
constexpr int kThreads = (1 + kIssuers + kEpiWarps) * 32;   // 19 warps, at most 96 registers a thread

struct IndexerParams {
    const float* w;
    const int32_t* q_pos0;
    const int32_t* kv_len;
    float* scores;
    int64_t ld;
    int B, L, Nmax;
    int G;        // query groups per batch
    int n_tiles;  // key tiles per batch row = ceil(Nmax / 128)
    int NC;       // key chunks per group
    int CH;       // key tiles per chunk
    int n_items;  // B * G * NC
    int32_t* status;  // device error word
    PageTable pages;  // paged key cache (pages.table == nullptr: dense [B][Nmax] rows)
    int box_rows;     // rows per key TMA box: 128 dense, min(page_size, 128) paged
};

template <int QG, int STAGES>
struct Cfg {
    static constexpr int N = QG * kHi;                      // MMA N
    static constexpr int A_HALF = kTileKeys * 64 * 2;       // 16 KB: 128 keys x 64 dims
    static constexpr int A_BYTES = 2 * A_HALF;              // 32 KB
    static constexpr int B_HALF = N * 64 * 2;               // N rows x 64 dims
    static constexpr int B_BYTES = 2 * B_HALF;
    static constexpr int NACC = (512 / N >= 4) ? 4 : 2;                 // TMEM accumulators in flight
    static constexpr int TMEM_COLS = (NACC * N < 32) ? 32 : NACC * N;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = STAGES * A_BYTES;
    static constexpr int OFF_BAR = OFF_B + B_BYTES;
    // barriers: a_full[S], a_empty[S], b_full, b_empty, acc_full[NACC], acc_empty[NACC]
    static constexpr int N_BARS = 2 * STAGES + 2 + 2 * NACC;
    static constexpr int OFF_TMEM = OFF_BAR + N_BARS * 8;
    static constexpr int OFF_ABORT = OFF_TMEM + 4;
    static constexpr int SMEM = OFF_ABORT + 4 + 1024;  // + slack for 1024-byte alignment
    static constexpr uint32_t IDESC = idesc_bf16_f32(kTileKeys, N, false, false);
};

constexpr int kChains = 2;   // independent packed FMA chains in the head sum (see weighted_relu_sum)
// One query's score for this thread's key: sum over the 32 heads of
// w[h] * relu(x[h]), x = the head's 32 TMEM columns, w in registers.  Even
// heads accumulate in .x and odd heads in .y of a packed f32x2 FMA; the two
// halves are added last.
__device__ __forceinline__ float weighted_relu_sum(const uint32_t (&x)[32], const float4 (&wv)[kHi / 4]) {
    // kChains independent packed chains: the epilogue, which paces this kernel, waits on the
    // dependent FMA sequence once per tile (16k chunk: one chain 300 us, two 285, four 289, eight
    // 306; the sums are exact on the integer-grid inputs, so the order changes no bit there)
    float2 s[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) s[c] = make_float2(0.f, 0.f);
#pragma unroll
    for (int h4 = 0; h4 < kHi / 4; ++h4) {
        float2& a = s[(2 * h4) % kChains];
        float2& b = s[(2 * h4 + 1) % kChains];
        a = __ffma2_rn(make_float2(wv[h4].x, wv[h4].y),
                       make_float2(fmaxf(__uint_as_float(x[4 * h4 + 0]), 0.f), fmaxf(__uint_as_float(x[4 * h4 + 1]), 0.f)), a);
        b = __ffma2_rn(make_float2(wv[h4].z, wv[h4].w),
                       make_float2(fmaxf(__uint_as_float(x[4 * h4 + 2]), 0.f), fmaxf(__uint_as_float(x[4 * h4 + 3]), 0.f)), b);
    }
#pragma unroll
    for (int w = kChains / 2; w >= 1; w /= 2)
#pragma unroll
        for (int c = 0; c < w; ++c) s[c] = make_float2(s[c].x + s[c + w].x, s[c].y + s[c + w].y);
    return s[0].x + s[0].y;
}

struct Item {
    int b, i0, nq, t_begin, t_end, n_comp_end;  // compute tiles are [t_begin, n_comp_end)
    int pos0, kl;
};

__device__ __forceinline__ Item decode_item(const IndexerParams& p, int item, int QG) {
    Item it;
    int c = item % p.NC;
    int bg = item / p.NC;
    int g = bg % p.G;
    it.b = bg / p.G;
    it.i0 = g * QG;
    it.nq = min(QG, p.L - it.i0);
    it.t_begin = c * p.CH;
    it.t_end = min(it.t_begin + p.CH, p.n_tiles);
    it.pos0 = __ldg(p.q_pos0 + it.b);
    it.kl = min(__ldg(p.kv_len + it.b), p.Nmax);
    long long lim_last = min((long long)it.pos0 + it.i0 + it.nq - 1, (long long)it.kl - 1);
    long long nk = lim_last < 0 ? 0 : lim_last + 1;  // keys [0, nk) have a causal query
    int comp_tiles = (int)((nk + kTileKeys - 1) / kTileKeys);
    it.n_comp_end = max(it.t_begin, min(it.t_end, comp_tiles));
    return it;
}

// The s-th item of this CTA (zig-zag over waves of gridDim.x items); -1 when done.
__device__ __forceinline__ int nth_item(const IndexerParams& p, int s) {
    int base = s * (int)gridDim.x;
    if (base >= p.n_items) return -1;
    int k = (s & 1) ? ((int)gridDim.x - 1 - (int)blockIdx.x) : (int)blockIdx.x;
    int item = base + k;
    return item < p.n_items ? item : -2;  // -2: no item in this wave for this CTA
}

template <int QG, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const IndexerParams p) {
    using C = Cfg<QG, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + C::OFF_A;
    uint8_t* sB = smem + C::OFF_B;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* a_full = bars;
    uint64_t* a_empty = bars + STAGES;
    uint64_t* b_full = bars + 2 * STAGES;
    uint64_t* b_empty = b_full + 1;
    uint64_t* acc_full = b_full + 2;
    uint64_t* acc_empty = b_full + 2 + C::NACC;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);

    const int warp = threadIdx.x / 32;
    const uint32_t lane = lane_id();

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&a_full[s], 1);
            mbar_init(&a_empty[s], 1);
        }
        mbar_init(b_full, 1);
        mbar_init(b_empty, kIssuers);   // each issuer's last MMA of an item has read the queries
        for (int a = 0; a < C::NACC; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], kEpiWarps * 32);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmap_q);
        tma_prefetch_desc(&tmap_k);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    griddep_wait();                 // inputs and outputs may belong to the previous kernel until here

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int it = 0, bi = 0;
            bool ok = true;
            for (int s = 0; ok; ++s) {
                int item = nth_item(p, s);
                if (item == -1) break;
                if (item < 0) continue;
                Item I = decode_item(p, item, QG);
                if (I.n_comp_end <= I.t_begin) continue;
                if (!(ok = mbar_wait_spin(b_empty, (bi & 1) ^ 1, abort_flag, p.status))) break;
                ++bi;
                mbar_arrive_expect_tx(b_full, C::B_BYTES);
                const int qrow = (I.b * p.L + I.i0) * kHi;
                tma_load_2d(sB, &tmap_q, b_full, 0, qrow);
                tma_load_2d(sB + C::B_HALF, &tmap_q, b_full, 64, qrow);
                for (int t = I.t_begin; t < I.n_comp_end; ++t, ++it) {
                    const int st = it % STAGES;
                    if (!(ok = mbar_wait_spin(&a_empty[st], ((it / STAGES) & 1) ^ 1, abort_flag, p.status))) break;
                    mbar_arrive_expect_tx(&a_full[st], C::A_BYTES);
                    uint8_t* dst = sA + st * C::A_BYTES;
                    if (p.pages.table == nullptr) {
                        const int krow = I.b * p.Nmax + t * kTileKeys;
                        tma_load_2d(dst, &tmap_k, &a_full[st], 0, krow);
                        tma_load_2d(dst + C::A_HALF, &tmap_k, &a_full[st], 64, krow);
                    } else {
                        // one box per page (or per 128 rows of a larger page); a box
                        // starts on a 1024-byte boundary, so the swizzled rows land
                        // exactly where one 128-row box would put them
                        for (int r = 0; r < kTileKeys; r += p.box_rows) {
                            const int j = t * kTileKeys + r;   // logical key of the box's first row
                            const int lp = j >> p.pages.shift;
                            int page = 0;
                            if (j < I.kl) {
                                page = __ldg(p.pages.table + (int64_t)I.b * p.pages.stride + lp);
                                if (page < 0 || page >= p.pages.num_pages) {
                                    raise_dev_error(p.status, DEV_ERR_BOUNDS);
                                    page = -1;   // a box wholly outside the pool: TMA fills zeros
                                }
                            }
                            const int krow = (page < 0) ? -p.box_rows
                                                        : (page << p.pages.shift) + (j & ((1 << p.pages.shift) - 1));
                            tma_load_2d(dst + r * 128, &tmap_k, &a_full[st], 0, krow);
                            tma_load_2d(dst + C::A_HALF + r * 128, &tmap_k, &a_full[st], 64, krow);
                        }
                    }
                }
            }
        }
    } else if (warp <= kIssuers) {
        // ------------------------------------------------------------ MMA issuers
        // Issuer i takes the key tiles whose running index is i mod kIssuers, so each stage and
        // each accumulator (both rings of even size) belongs to one issuer, and one issuer's
        // barrier waits overlap the other's MMAs.  Descriptors are precomputed bases plus
        // compile-time offsets added to the low word (shared addresses < 256 KB cannot carry).
        // (Measured: 305 -> 300 us at the 16k chunk; the N = 128 MMAs of this GEMM already ran
        // close to the tensor rate with one issuer, unlike the attention's N = 64 ones.)
        static_assert(STAGES % kIssuers == 0 && C::NACC % kIssuers == 0, "rings split evenly over the issuers");
        const int iss = warp - 1;
        if (lane == 0) {
            int it = 0, bi = 0, acc_it = 0;
            bool ok = true;
            const uint64_t a_desc = sdesc_sw128(smem_u32(sA), 16, 1024);
            const uint64_t b_desc = sdesc_sw128(smem_u32(sB), 16, 1024);
            const uint32_t a_hi = (uint32_t)(a_desc >> 32), b_hi = (uint32_t)(b_desc >> 32);
            const uint32_t b_lo = (uint32_t)b_desc;
            for (int s = 0; ok; ++s) {
                int item = nth_item(p, s);
                if (item == -1) break;
                if (item < 0) continue;
                Item I = decode_item(p, item, QG);
                if (I.n_comp_end <= I.t_begin) continue;
                if (!(ok = mbar_wait_spin(b_full, bi & 1, abort_flag, p.status))) break;
                ++bi;
                tc_fence_after();
                for (int t = I.t_begin; t < I.n_comp_end; ++t, ++it, ++acc_it) {
                    if (it % kIssuers != iss) continue;
                    const int st = it % STAGES;
                    const int acc = acc_it % C::NACC;
                    if (!(ok = mbar_wait_spin(&a_full[st], (it / STAGES) & 1, abort_flag, p.status))) break;
                    if (!(ok = mbar_wait_spin(&acc_empty[acc], ((acc_it / C::NACC) & 1) ^ 1, abort_flag, p.status))) break;
                    tc_fence_after();
                    const uint32_t a_lo = (uint32_t)a_desc + (uint32_t)(st * (C::A_BYTES >> 4));
                    const uint32_t d = tmem_base + acc * C::N;
#pragma unroll
                    for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_bf16_ss_lo(d, a_lo + (uint32_t)(kb * (C::A_HALF >> 4) + 2 * kk), a_hi,
                                           b_lo + (uint32_t)(kb * (C::B_HALF >> 4) + 2 * kk), b_hi, C::IDESC,
                                           (kb | kk) != 0);
                    }
                    mma_commit(&a_empty[st]);
                    mma_commit(&acc_full[acc]);
                }
                if (ok) mma_commit(b_empty);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 1 + kIssuers ..)
        // kEpiWarps / 4 warps per TMEM lane quadrant, one of the group's queries
        // each (warps whose query is past the group's end only write -inf).
        static_assert(QG <= kEpiWarps / 4, "one query per epilogue warp");
        const int e = warp - 1 - kIssuers;           // 0..kEpiWarps-1
        const int quad = warp & 3;                   // TMEM lane quadrant of this warp
        const int q = e >> 2;                        // this warp's query within the group
        const int key_in_tile = quad * 32 + (int)lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        int acc_it = 0;
        bool ok = true;
        for (int s = 0; ok; ++s) {
            int item = nth_item(p, s);
            if (item == -1) break;
            if (item < 0) continue;
            Item I = decode_item(p, item, QG);
            const int64_t row0 = (int64_t)I.b * p.L + I.i0;
            const bool mine = q < I.nq;               // warp-uniform
            // the query's 32 head weights, in registers for the whole item
            float4 wq[kHi / 4];
            {
                const float4* w4 = reinterpret_cast<const float4*>(p.w + (row0 + q) * kHi);
#pragma unroll
                for (int h4 = 0; h4 < kHi / 4; ++h4) wq[h4] = mine ? __ldg(w4 + h4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            const int lim = (int)min((long long)I.pos0 + I.i0 + q, (long long)I.kl - 1);   // last causal key
            float* srow_item = p.scores + (row0 + q) * p.ld + key_in_tile;
            for (int t = I.t_begin; t < I.t_end; ++t) {
                const int j = t * kTileKeys + key_in_tile;
                float* srow = srow_item + t * kTileKeys;
                if (t < I.n_comp_end) {
                    const int acc = acc_it % C::NACC;
                    // warp-uniform outcome: the TMEM load below is warp-collective
                    // polled rather than suspended: the epilogue paces the kernel, and a suspended
                    // try_wait resumes later (285 -> 283 us at 16k, 1189 -> 1174 us at 64k)
                    ok = __all_sync(0xffffffffu, mbar_wait_spin(&acc_full[acc], (acc_it / C::NACC) & 1, abort_flag, p.status));
                    if (!ok) break;
                    tc_fence_after();
                    if (q < QG) {   // warp-uniform: TMEM columns of this query exist
                        uint32_t v[32];
                        tmem_ld32(tmem_base + lane_addr + acc * C::N + q * kHi, v);
                        tmem_ld_wait();
                        const float r = weighted_relu_sum(v, wq);
                        if (j < p.Nmax && mine) *srow = (j <= lim) ? r : -INFINITY;
                    }
                    tc_fence_before();
                    mbar_arrive(&acc_empty[acc]);
                    ++acc_it;
                } else if (j < p.Nmax && mine) {
                    *srow = -INFINITY;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int QG, int STAGES>
dsa_status_t launch_impl(const void* q_idx, const void* k_idx, const IndexerParams& prm, int B, int L, int Nmax,
                         cudaStream_t stream) {
    using C = Cfg<QG, STAGES>;
    CUtensorMap tq, tk;
    dsa_status_t st;
    if ((st = make_tmap_bf16_2d(&tq, q_idx, kDi, (uint64_t)B * L * kHi, kDi * 2, 64, QG * kHi)) != DSA_OK) return st;
    const uint64_t k_rows = prm.pages.table ? ((uint64_t)prm.pages.num_pages << prm.pages.shift) : (uint64_t)B * Nmax;
    if ((st = make_tmap_bf16_2d(&tk, k_idx, kDi, k_rows, kDi * 2, 64, prm.box_rows)) != DSA_OK) return st;
    auto kern = indexer_kernel<QG, STAGES>;
    if ((st = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::SMEM)) != DSA_OK) return st;
    int grid = min(prm.n_items, device_sm_count());
    if (launch_pdl(kern, dim3(grid), dim3(kThreads), C::SMEM, stream, tq, tk, prm) != cudaSuccess) return DSA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace

dsa_status_t launch_indexer(const void* q_idx, const void* k_idx, const float* w, const int32_t* q_pos0,
                            const int32_t* kv_len, int B, int L, int Nmax, float* scores, int64_t ld,
                            const PageTable& pages, cudaStream_t stream) {
    const int QG = (L == 1) ? 1 : 4;
    IndexerParams p;
    p.w = w;
    p.q_pos0 = q_pos0;
    p.kv_len = kv_len;
    p.scores = scores;
    p.ld = ld;
    p.B = B;
    p.L = L;
    p.Nmax = Nmax;
    p.G = ceil_div(L, QG);
    p.n_tiles = ceil_div(Nmax, kTileKeys);
    const int sms = device_sm_count();
    // Enough items for a few per CTA (load balance), long chunks otherwise
    // (the group's queries are loaded once per item).
    const long long groups = (long long)B * p.G;
    long long nc = (4LL * sms + groups - 1) / groups;
    // A call of at most two tiles per SM (batched decode) is latency bound: one round of items
    // (about one per SM, their tiles pipelined) beats several rounds of one-tile items.
    if (groups * p.n_tiles <= 2LL * sms) nc = sms / groups;
    if (nc < 1) nc = 1;
    if (nc > p.n_tiles) nc = p.n_tiles;
    p.CH = ceil_div(p.n_tiles, (int)nc);
    p.NC = ceil_div(p.n_tiles, p.CH);
    long long items = groups * p.NC;
    if (items > 0x7FFFFFFFLL) return DSA_ERR_UNSUPPORTED_SHAPE;
    p.n_items = (int)items;
    p.status = device_status_ptr();
    p.pages = pages;
    p.box_rows = pages.table ? (pages.shift >= 7 ? kTileKeys : (1 << pages.shift)) : kTileKeys;
    if (QG == 4) return launch_impl<4, 4>(q_idx, k_idx, p, B, L, Nmax, stream);
    return launch_impl<1, 4>(q_idx, k_idx, p, B, L, Nmax, stream);
}

}  // namespace dsa
