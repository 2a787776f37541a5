// topk.cu -- per-query top-k key selection over float32 indexer scores.
//
// What it computes (exo PR #2539, section "Prefill": each query keeps its
// index_topk = 2048 best keys; bullet "The first 2048 queries attend causally":
// a query with n <= top_k causal keys keeps all of them).  Readings of what the
// pages leave open: equal scores rank the lower key index first, -0.0 equals
// +0.0, the selection is written in ascending key order and unused slots hold -1.
//
// How: one CTA per score row runs an exact radix select.
//   * Scores map to order-preserving 32-bit keys (-0.0 folded onto +0.0).
//   * Up to three histogram passes (12 + 12 + 8 bits, shared-memory atomics)
//     narrow down the threshold key T and how many keys equal to T are still
//     needed; a pass is skipped as soon as the threshold bucket is taken whole.
//   * A final pass walks the row in index order and compacts the chosen keys
//     with block-wide prefix sums: every key above T, plus the first `need`
//     keys equal to T (this is the lower-index tie rule).  Positions come from
//     the prefix sums, so the output is ascending without a sort.
//   * Calls with Nmax <= 4096 (512 threads of eight keys, four CTAs per SM)
//     and 8192 < Nmax <= 16384 (1024 threads of 16 keys, two CTAs per SM): a thread
//     holds a contiguous run of keys of the row in registers, loaded once from
//     HBM with all of its loads in flight, for every pass; one block scan
//     orders the compaction.
//   * Other sizes stream the row on every pass (the first pass reads HBM, later
//     passes mostly hit L2) with four CTAs per SM: the passes are latency
//     bound, and more rows in flight win for short rows, while long rows do
//     not fit in registers.  For long rows a thread keeps four float4 loads in
//     flight per histogram step and compacts a run of eight float4 per block
//     scan (64k keys: 0.90 -> 0.69 ms for 4096 rows on GB300).  Rows of at least
//     32768 keys first take a lower bound for the threshold bucket from an
//     eighth of the row and copy every key above it into a shared-memory list
//     in one read; the full histogram pass runs only when that list misses.
#include <cuda_runtime.h>

#include <cstdint>

#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 4096;

struct TopkParams {
    const float* scores;
    int64_t ld;
    const int32_t* q_pos0;
    const int32_t* kv_len;
    int32_t* idx;
    int B, L, Nmax, K;
};

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;  // -0.0 == +0.0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive scan of one uint32 per thread (NT threads); returns the
// exclusive prefix and writes the block total to *total.  Uses
// warp_sums[NT / 32 + 1].
template <int NT = kThreads>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* warp_sums, uint32_t* total) {
    constexpr int kWarps = NT / 32;
    static_assert(kWarps <= 32, "one warp scans the warp sums");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t s = lane < kWarps ? warp_sums[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < kWarps) warp_sums[lane] = s;  // inclusive over warps
        if (lane == kWarps - 1) warp_sums[kWarps] = s;
    }
    __syncthreads();
    uint32_t excl = x - v + (warp > 0 ? warp_sums[warp - 1] : 0u);
    *total = warp_sums[kWarps];
    __syncthreads();
    return excl;
}

// Given hist[nbins] of the still-tied keys and `need` (>= 1, <= their count),
// find the bin B* (scanning from the largest bin down) holding the need-th
// largest key.  Writes sel[0] = B*, sel[1] = need minus the keys in bins above.
template <int NT = kThreads>
__device__ void find_bin(const uint32_t* hist, int nbins, uint32_t need, uint32_t* warp_sums, uint32_t* sel) {
    const int per = nbins / NT;  // 8 for 4096 bins and 512 threads; 0 for 256 bins (then one bin a thread)
    uint32_t local = 0;
    const int t = threadIdx.x;
    const bool active = (per > 0) ? true : (t < nbins);
    const int p = per > 0 ? per : 1;
    // thread t owns bins (from the top) [t*p, t*p + p)
    if (active)
        for (int k = 0; k < p; ++k) local += hist[nbins - 1 - (t * p + k)];
    uint32_t total;
    uint32_t above = block_excl_scan<NT>(local, warp_sums, &total);
    if (active && above < need && above + local >= need) {
        uint32_t run = above;
        for (int k = 0; k < p; ++k) {
            int bin = nbins - 1 - (t * p + k);
            uint32_t c = hist[bin];
            if (run + c >= need) {
                sel[0] = (uint32_t)bin;
                sel[1] = need - run;
                sel[2] = c;  // keys in the threshold bin
                break;
            }
            run += c;
        }
    }
    __syncthreads();
}

// Number of causal keys of score row r (query i of batch b at q_pos0[b] + i).
__device__ __forceinline__ int row_keys(const TopkParams& p, int r) {
    const int b = r / p.L, i = r % p.L;
    const long long pos = (long long)__ldg(p.q_pos0 + b) + i;
    const long long kl = min((long long)__ldg(p.kv_len + b), (long long)p.Nmax);
    return (int)max(0LL, min(pos + 1, kl));
}

// 8192 < Nmax <= 16384: 1024 threads of 16 keys each, two CTAs per SM (512 threads of 32 keys: 3%
// slower on GB300).
constexpr int kLongRowThreads = 1024;
constexpr int kPer = 16;                              // keys a thread holds: a contiguous run of the row
constexpr int kChunk = kLongRowThreads * kPer;        // 16384 keys: the longest register-resident row
// Below this many keys a row is short enough that four streaming CTAs per SM
// (more rows in flight) beat two register-resident ones (measured on GB300).
constexpr int kRegMinKeys = 8192;
// Rows of at most 4096 keys: eight keys a thread (one 512-thread block holds the
// row in registers) at four CTAs per SM beat the streaming kernel (GB300: 4096
// rows of the first 4k chunk 48.8 -> 41.6 us, a batch-8 decode step's 13 -> 11 us).
constexpr int kShortPer = 8;
constexpr int kShortKeys = kThreads * kShortPer;
// Streaming kernel shapes: kU = float4 loads a thread keeps in flight in a
// histogram pass, kC = float4 a thread compacts per block scan (4 kC <= 32 mask
// bits).  Long rows take (4, 8); short rows (one or two block steps) are faster
// with (1, 1), where every thread has data in every step (measured on GB300).
constexpr int kLongU = 4, kLongC = 8;

// Load this thread's run of the row (keys PER t .. PER t + PER - 1) as order
// keys; positions past the row get key 0 (no finite or infinite score maps to
// 0).  The float4 loads are issued together and go through L1, which keeps the
// 128-byte lines the warp's strided accesses touch.
template <int PER>
__device__ __forceinline__ void load_run(const float4* row4, int n, uint32_t (&key)[PER]) {
    const int v0 = threadIdx.x * (PER / 4);
    const int n4 = (n + 3) / 4;
    float4 f[PER / 4];
#pragma unroll
    for (int c = 0; c < PER / 4; ++c) f[c] = (v0 + c < n4) ? __ldg(row4 + v0 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = 0; c < PER / 4; ++c) {
        const float e[4] = {f[c].x, f[c].y, f[c].z, f[c].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) key[4 * c + k] = (4 * (v0 + c) + k < n) ? order_key(e[k]) : 0u;
    }
}

// Long rows, after the first histogram pass fixed the top 12 bits (bucket b1)
// of the threshold: if the keys at or above b1 number at most kCap, one more
// read of the row copies them (order key and index, in ascending index order)
// into shared memory, and the rest of the selection runs there.  Two reads of
// the row instead of up to four.
constexpr int kCap = 4608;
constexpr int kCapPer = kCap / kThreads;    // 9 list entries a thread orders in the final scan
// Rows of at least this many keys start from a sampled lower bound (n / 8 keys
// sampled, so the sample's target rank stays well inside it for top_k <= 2048).
constexpr int kSampleMinKeys = 32768;
static_assert(kCap % kThreads == 0 && kCapPer <= 32, "final scan: one mask bit per entry");

//
// With `bound` set, b1 is only a lower bound for the threshold bucket (from a
// sample of the row): the list then holds every key whose top 12 bits are at
// least b1, the selection starts from the full key, and the call returns false
// (nothing written) when the list came out shorter than K (the bound was too
// high) or longer than kCap.  Returns true once the row's indices are written.
__device__ bool collect_and_select(const float4* row4, int n, int n4, uint32_t b1, uint32_t need, int K,
                                   int32_t* out, uint32_t* hist, uint32_t* warp_sums, uint32_t* sel,
                                   uint32_t* c_key, int32_t* c_idx, bool bound) {
    const int tid = threadIdx.x;
    // ---- copy keys with top-12 bits >= b1, two coalesced float4 per thread per block step;
    // one scan of (count of float4 0) | (count of float4 1) << 16 orders both.
    uint32_t base = 0;
    for (int base4 = 0; base4 < n4; base4 += 2 * kThreads) {
        float4 f[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int v = base4 + u * kThreads + tid;
            f[u] = (v < n4) ? __ldcg(row4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        uint32_t key[2][4];
        uint32_t m[2] = {0u, 0u};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int v = base4 + u * kThreads + tid;
            const float e[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                key[u][k] = order_key(e[k]);
                if (4 * v + k < n && (key[u][k] >> 20) >= b1) m[u] |= 1u << k;
            }
        }
        uint32_t total;
        const uint32_t pre = block_excl_scan((uint32_t)__popc(m[0]) | ((uint32_t)__popc(m[1]) << 16), warp_sums, &total);
        uint32_t pos[2] = {base + (pre & 0xFFFFu), base + (total & 0xFFFFu) + (pre >> 16)};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int v = base4 + u * kThreads + tid;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if ((m[u] & (1u << k)) && pos[u] < (uint32_t)kCap) {   // the count fits by the histogram
                    c_key[pos[u]] = key[u][k];
                    c_idx[pos[u]] = 4 * v + k;
                    ++pos[u];
                }
            }
        }
        base += (total & 0xFFFFu) + (total >> 16);
    }
    if (bound && (base < (uint32_t)K || base > (uint32_t)kCap)) return false;   // base is block-uniform
    const int M = min((int)base, kCap);   // = keys above b1 + keys in b1 <= kCap
    // ---- refine the threshold among the bucket's keys (bits 19..8, then 7..0); from a bound,
    // first find the bucket among the list (bits 31..20)
    uint32_t prefix = bound ? 0u : b1;
    int shift = bound ? 32 : 20;
    if (bound) need = (uint32_t)K;
    for (int pass = bound ? 0 : 1; pass < 3; ++pass) {
        const int bits = (pass == 2) ? 8 : 12;
        const int nbins = 1 << bits;
        const int new_shift = shift - bits;
        for (int k = tid; k < nbins; k += kThreads) hist[k] = 0u;
        __syncthreads();
        for (int e = tid; e < M; e += kThreads) {
            const uint32_t kk = c_key[e];
            if (shift == 32 || (kk >> shift) == prefix) atomicAdd(&hist[(kk >> new_shift) & (uint32_t)(nbins - 1)], 1u);
        }
        __syncthreads();
        find_bin(hist, nbins, need, warp_sums, sel);
        const uint32_t bin = sel[0], rem = sel[1], cnt = sel[2];
        prefix = (shift == 32 ? 0u : (prefix << bits)) | bin;
        shift = new_shift;
        need = rem;
        __syncthreads();
        if (rem == cnt) break;
    }
    // ---- ordered selection over the list: every key above the class, then the first `need` of it
    uint32_t gmask = 0, emask = 0;
    const int e0 = tid * kCapPer;
#pragma unroll
    for (int q = 0; q < kCapPer; ++q) {
        if (e0 + q < M) {
            const uint32_t sk = c_key[e0 + q] >> shift;
            if (sk > prefix) gmask |= 1u << q;
            else if (sk == prefix) emask |= 1u << q;
        }
    }
    uint32_t total;
    const uint32_t pre = block_excl_scan(((uint32_t)__popc(emask) << 16) | (uint32_t)__popc(gmask), warp_sums, &total);
    uint32_t g_before = pre & 0xFFFFu;
    uint32_t e_before = pre >> 16;
    while (gmask | emask) {
        const int q = __ffs(gmask | emask) - 1;
        const uint32_t bit = 1u << q;
        const int j = c_idx[e0 + q];
        if (gmask & bit) {
            const uint32_t pos = g_before + min(need, e_before);
            if (pos < (uint32_t)K) out[pos] = j;
            ++g_before;
        } else {
            if (e_before < need && g_before + e_before < (uint32_t)K) out[g_before + e_before] = j;
            ++e_before;
        }
        gmask &= ~bit;
        emask &= ~bit;
    }
    __syncthreads();   // the list and the histogram are reused by the next row
    return true;
}

// Streaming select (any row length): four CTAs per SM; every pass reads the
// row again (the first from HBM, later ones mostly from L2).
template <int kU, int kC, bool kCollect>
__global__ void __launch_bounds__(kThreads, 4) topk_stream_kernel(const TopkParams p) {
    __shared__ uint32_t hist[kBins];
    __shared__ uint32_t warp_sums[kWarps + 1];
    __shared__ uint32_t sel[3];
    extern __shared__ uint32_t dyn_smem[];           // kCollect: the candidate list (ascending key index)
    uint32_t* c_key = dyn_smem;
    int32_t* c_idx = reinterpret_cast<int32_t*>(dyn_smem + kCap);

    griddep_wait();                 // the scores may still be written by the previous kernel
    const int R = p.B * p.L;
    for (int r = blockIdx.x; r < R; r += gridDim.x) {
        const int b = r / p.L, i = r % p.L;
        const long long pos = (long long)__ldg(p.q_pos0 + b) + i;
        const long long kl = min((long long)__ldg(p.kv_len + b), (long long)p.Nmax);
        long long n_ll = min(pos + 1, kl);
        const int n = (int)max(0LL, n_ll);
        int32_t* out = p.idx + (int64_t)r * p.K;
        if (n <= p.K) {
            for (int t = threadIdx.x; t < p.K; t += kThreads) out[t] = t < n ? t : -1;
            continue;
        }
        const float* row = p.scores + (int64_t)r * p.ld;
        const float4* row4 = reinterpret_cast<const float4*>(row);
        const int n4 = (n + 3) / 4;

        if (kCollect && n >= kSampleMinKeys) {
            // ---- a lower bound for the threshold bucket from every eighth 128-byte line of the
            // row (n / 8 keys): the bucket holding the sample's (9 K / 64 + 24)-th largest key,
            // about 3.5 standard deviations past its expected K / 8 at K = 2048; then one read of
            // the row copies every key from that bucket up (instead of a full histogram read first)
            for (int k = threadIdx.x; k < kBins; k += kThreads) hist[k] = 0u;
            __syncthreads();
            const int s_f4 = ((n4 + 63) / 64) * 8;   // float4 0..7 of every 64
            for (int sidx = threadIdx.x; sidx < s_f4; sidx += kThreads) {
                const int v = 64 * (sidx >> 3) + (sidx & 7);
                if (v < n4) {
                    const float4 f = __ldcg(row4 + v);
                    const float e[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (4 * v + k < n) atomicAdd(&hist[order_key(e[k]) >> 20], 1u);
                }
            }
            __syncthreads();
            find_bin(hist, kBins, (uint32_t)(p.K + p.K / 8 + 8 * 24) / 8u, warp_sums, sel);
            const uint32_t b_lo = sel[0];
            __syncthreads();
            if (collect_and_select(row4, n, n4, b_lo, 0u, p.K, out, hist, warp_sums, sel, c_key, c_idx, true))
                continue;
            __syncthreads();   // fall back to the full passes
        }

        // ---- radix narrowing: (shift, prefix, need) describe the threshold class
        int shift = 32;        // keys compared on bits [shift, 32); 32 = nothing fixed yet
        uint32_t prefix = 0;
        uint32_t need = (uint32_t)p.K;
        bool collected = false;
        const int digit_bits[3] = {12, 12, 8};
        for (int pass = 0; pass < 3; ++pass) {
            const int bits = digit_bits[pass];
            const int nbins = 1 << bits;
            const int new_shift = shift - bits;
            for (int k = threadIdx.x; k < nbins; k += kThreads) hist[k] = 0u;
            __syncthreads();
            for (int v0 = threadIdx.x; v0 < n4; v0 += kThreads * kU) {
                float4 f[kU];   // kU coalesced loads in flight before any is used
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int v = v0 + u * kThreads;
                    f[u] = (v < n4) ? __ldcg(row4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int v = v0 + u * kThreads;
                    const float e[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        if (4 * v + k < n) {
                            const uint32_t key = order_key(e[k]);
                            const bool in_class = (shift == 32) || ((key >> shift) == prefix);
                            if (in_class) atomicAdd(&hist[(key >> new_shift) & (uint32_t)(nbins - 1)], 1u);
                        }
                    }
                }
            }
            __syncthreads();
            find_bin(hist, nbins, need, warp_sums, sel);
            const uint32_t bin = sel[0], rem = sel[1], cnt = sel[2];
            prefix = (shift == 32 ? 0u : (prefix << bits)) | bin;
            shift = new_shift;
            need = rem;
            __syncthreads();
            if (rem == cnt) break;  // the whole threshold bucket is taken
            if (kCollect && pass == 0 && (uint32_t)p.K - rem + cnt <= (uint32_t)kCap) {
                collected = true;   // block-uniform: sel[] is shared
                break;
            }
        }
        if (kCollect && collected) {
            collect_and_select(row4, n, n4, prefix, need, p.K, out, hist, warp_sums, sel, c_key, c_idx, false);
            continue;
        }

        // ---- ordered compaction: keys above the class, then the first `need` of the class.
        // A thread takes a contiguous run of kC float4 per block step (loads through L1,
        // which keeps the lines of the warp's strided accesses), so one block scan orders
        // 4 kC keys per thread.
        uint32_t g_base = 0, e_base = 0;
        for (int base4 = 0; base4 < n4; base4 += kThreads * kC) {
            const int v0 = base4 + threadIdx.x * kC;
            float4 f[kC];
#pragma unroll
            for (int u = 0; u < kC; ++u) f[u] = (v0 + u < n4) ? __ldg(row4 + v0 + u) : make_float4(0.f, 0.f, 0.f, 0.f);
            uint32_t gmask = 0, emask = 0;   // bit 4 u + k: key 4 (v0 + u) + k
#pragma unroll
            for (int u = 0; u < kC; ++u) {
                const float e[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (4 * (v0 + u) + k < n) {
                        const uint32_t key = order_key(e[k]) >> shift;
                        if (key > prefix) gmask |= 1u << (4 * u + k);
                        else if (key == prefix) emask |= 1u << (4 * u + k);
                    }
                }
            }
            const uint32_t packed = ((uint32_t)__popc(emask) << 16) | (uint32_t)__popc(gmask);
            uint32_t total;
            const uint32_t pre = block_excl_scan(packed, warp_sums, &total);
            uint32_t g_before = g_base + (pre & 0xFFFFu);
            uint32_t e_before = e_base + (pre >> 16);
            while (gmask | emask) {
                const int k = __ffs(gmask | emask) - 1;
                const uint32_t bit = 1u << k;
                const int j = 4 * v0 + k;
                if (gmask & bit) {
                    const uint32_t pos = g_before + min(need, e_before);
                    if (pos < (uint32_t)p.K) out[pos] = j;
                    ++g_before;
                } else {
                    if (e_before < need && g_before + e_before < (uint32_t)p.K) out[g_before + e_before] = j;
                    ++e_before;
                }
                gmask &= ~bit;
                emask &= ~bit;
            }
            g_base += total & 0xFFFFu;
            e_base += total >> 16;
        }
        __syncthreads();
    }
}

// Register-resident select for rows of up to one chunk (16384 keys): the row
// is loaded once and stays in registers for every pass (two CTAs per SM).
template <int PER, int MINB, int NT = kThreads>
__global__ void __launch_bounds__(NT, MINB) topk_reg_kernel(const TopkParams p) {
    __shared__ uint32_t hist[kBins];
    __shared__ uint32_t warp_sums[NT / 32 + 1];
    __shared__ uint32_t sel[3];

    griddep_wait();                 // the scores may still be written by the previous kernel
    const int R = p.B * p.L;
    for (int r = blockIdx.x; r < R; r += gridDim.x) {
        const int n = row_keys(p, r);
        int32_t* out = p.idx + (int64_t)r * p.K;
        if (n <= p.K) {
            for (int t = threadIdx.x; t < p.K; t += NT) out[t] = t < n ? t : -1;
            continue;
        }
        const float4* row4 = reinterpret_cast<const float4*>(p.scores + (int64_t)r * p.ld);
        uint32_t key[PER];
        load_run<PER>(row4, n, key);

        // ---- radix narrowing: (shift, prefix, need) describe the threshold class
        int shift = 32;        // keys compared on bits [shift, 32); 32 = nothing fixed yet
        uint32_t prefix = 0;
        uint32_t need = (uint32_t)p.K;
        const int digit_bits[3] = {12, 12, 8};
        for (int pass = 0; pass < 3; ++pass) {
            const int bits = digit_bits[pass];
            const int nbins = 1 << bits;
            const int new_shift = shift - bits;
            for (int k = threadIdx.x; k < nbins; k += NT) hist[k] = 0u;
            __syncthreads();
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const uint32_t kk = key[k];
                const bool in_class = (shift == 32) || ((kk >> shift) == prefix);
                if (kk != 0u && in_class) atomicAdd(&hist[(kk >> new_shift) & (uint32_t)(nbins - 1)], 1u);
            }
            __syncthreads();
            find_bin<NT>(hist, nbins, need, warp_sums, sel);
            const uint32_t bin = sel[0], rem = sel[1], cnt = sel[2];
            prefix = (shift == 32 ? 0u : (prefix << bits)) | bin;
            shift = new_shift;
            need = rem;
            __syncthreads();
            if (rem == cnt) break;  // the whole threshold bucket is taken
        }

        // ---- ordered compaction: keys above the class, then the first `need` of the class.
        // One block scan orders every thread's contiguous run.
        {
            uint32_t gmask = 0, emask = 0;
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const uint32_t kk = key[k];
                const uint32_t sk = kk >> shift;
                if (kk != 0u && sk > prefix) gmask |= 1u << k;
                else if (kk != 0u && sk == prefix) emask |= 1u << k;
            }
            const uint32_t packed = ((uint32_t)__popc(emask) << 16) | (uint32_t)__popc(gmask);
            uint32_t total;
            const uint32_t pre = block_excl_scan<NT>(packed, warp_sums, &total);
            (void)total;
            uint32_t g_before = pre & 0xFFFFu;
            uint32_t e_before = pre >> 16;
            const int j0 = threadIdx.x * PER;
            while (gmask | emask) {
                const int k = __ffs(gmask | emask) - 1;
                const uint32_t bit = 1u << k;
                if (gmask & bit) {
                    const uint32_t pos = g_before + min(need, e_before);
                    if (pos < (uint32_t)p.K) out[pos] = j0 + k;
                    ++g_before;
                } else {
                    if (e_before < need && g_before + e_before < (uint32_t)p.K) out[g_before + e_before] = j0 + k;
                    ++e_before;
                }
                gmask &= ~bit;
                emask &= ~bit;
            }
        }
        __syncthreads();
    }
}

}  // namespace

dsa_status_t launch_topk(const float* scores, int64_t ld, const int32_t* q_pos0, const int32_t* kv_len, int B,
                         int L, int Nmax, int top_k, int32_t* idx, cudaStream_t stream) {
    TopkParams p{scores, ld, q_pos0, kv_len, idx, B, L, Nmax, top_k};
    const long long R = (long long)B * L;
    if (Nmax <= kShortKeys) {
        const int grid = (int)min(R, (long long)device_sm_count() * 4);
        if (launch_pdl(topk_reg_kernel<kShortPer, 4>, dim3(grid), dim3(kThreads), 0, stream, p) != cudaSuccess)
            return DSA_ERR_CUDA;
    } else if (Nmax > kRegMinKeys && Nmax <= kChunk) {
        const int grid = (int)min(R, (long long)device_sm_count() * 2);
        if (launch_pdl(topk_reg_kernel<kPer, 2, kLongRowThreads>, dim3(grid), dim3(kLongRowThreads), 0, stream, p) !=
            cudaSuccess)
            return DSA_ERR_CUDA;
    } else {
        const int grid = (int)min(R, (long long)device_sm_count() * 4);
        cudaError_t e;
        if (Nmax > kChunk) {
            auto kern = topk_stream_kernel<kLongU, kLongC, true>;
            constexpr int list_bytes = kCap * 8;   // candidate keys and indices
            dsa_status_t st = ensure_smem_attr(reinterpret_cast<const void*>(kern), list_bytes);
            if (st != DSA_OK) return st;
            e = launch_pdl(kern, dim3(grid), dim3(kThreads), list_bytes, stream, p);
        } else {
            e = launch_pdl(topk_stream_kernel<1, 1, false>, dim3(grid), dim3(kThreads), 0, stream, p);
        }
        if (e != cudaSuccess) return DSA_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
