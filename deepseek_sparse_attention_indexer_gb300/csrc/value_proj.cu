// value_proj.cu -- the value up-projection that follows sparse absorbed-MLA attention.
//
// What it computes (SlimServe "GLM52_PIPELINE_TRACE.md", section 6 "Attention
// core (absorbed MLA)": after V.softmax over the 512-wide latent, the product
// with wv_b turns each head's latent output into that head's value, the
// "MQA -> MHA" decompression; Config line: kv_lora_rank 512, v_head_dim 256,
// 64 heads.  exo PR #2539, section "Prefill": the value up-projection runs once
// for all queries of a chunk instead of once per query block):
//   v[r, h, e] = sum_{d < 512} o[r, h, d] * wv_b[h, e, d],   e < 256,
// bf16 inputs, float32 accumulation, bf16 output (round to nearest even).
//
// How (GB300 design):
//   * One tcgen05 GEMM tile per (head h, block of 128 rows): M = 128 rows of o
//     (A operand, TMA boxes of the strided [R, 64 * 512] view, so no copy of
//     the head's slice is ever made), N = 256 output features (the head's whole
//     wv_b slice, K-major exactly as stored), K = 512 in eight 64-wide blocks
//     streamed through a 4-stage TMA ring (16 KB of o + 32 KB of weights a
//     stage).  N = 256 keeps every MMA at the full dense rate.
//   * Two 256-column TMEM accumulators: the epilogue of one tile overlaps the
//     MMAs of the next.  Each epilogue warp converts its 32 rows x 64 columns at
//     a time to bf16 in a 128-byte-swizzled shared-memory block and writes it
//     with one TMA tile store: HBM gets whole 128-byte lines from the copy
//     engine instead of 16-byte stores spread over 32 rows 32 KB apart (those
//     stores cost 23 us of the 89 us the kernel took at 4096 rows).
//   * Persistent CTAs walk the tiles head-fastest, so the CTAs in flight share
//     the 16 MB of weights through L2 and each row of o is read from HBM once.
//   * The kernel is bound by HBM: per (row, head) it moves 1024 bytes of o in
//     and 512 bytes of v out for 262,144 FLOP (about 170 FLOP a byte, below the
//     ~280 FLOP/byte ridge of GB300's measured bf16 peak over its HBM copy rate).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {

namespace {

constexpr int kH = DSA_HEADS;          // 64
constexpr int kDv = DSA_V_DIM;         // 512 (K)
constexpr int kE = DSA_V_HEAD_DIM;     // 256 (N)
constexpr int kBM = 128;               // rows per tile (M)
constexpr int kKB = kDv / 64;          // 8 K-blocks of 64
constexpr int kStages = 4;
constexpr int kABytes = kBM * 128;     // 16 KB: 128 rows x 64 dims
constexpr int kBBytes = kE * 128;      // 32 KB: 256 features x 64 dims
constexpr int kEpiWarps = 8;           // two per TMEM lane quadrant, 128 columns each
constexpr int kThreads = (2 + kEpiWarps) * 32;

constexpr int kStgBytes = 32 * 128;    // 4 KB a warp: 32 rows x 64 bf16, one TMA store box

constexpr int OFF_A = 0;
constexpr int OFF_B = kStages * kABytes;
constexpr int OFF_STG = OFF_B + kStages * kBBytes;
constexpr int OFF_BAR = OFF_STG + kEpiWarps * kStgBytes;
// barriers: full[S], empty[S], acc_full[2], acc_empty[2]
constexpr int N_BARS = 2 * kStages + 4;
constexpr int OFF_TMEM = OFF_BAR + N_BARS * 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int SMEM_BYTES = OFF_ABORT + 4 + 1024;   // + slack for the 1024-byte alignment
constexpr uint32_t TMEM_COLS = 2 * kE;             // 512
constexpr uint32_t IDESC = idesc_bf16_f32(kBM, kE, false, false);
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

struct VprojParams {
    int R;
    int n_units;        // 64 * ceil(R / 128)
    int32_t* status;    // device error word
};

__global__ void __launch_bounds__(kThreads, 1)
    value_up_proj_kernel(const __grid_constant__ CUtensorMap tmap_o, const __grid_constant__ CUtensorMap tmap_w,
                         const __grid_constant__ CUtensorMap tmap_v, const VprojParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + OFF_A;
    uint8_t* sB = smem + OFF_B;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    uint64_t* acc_full = bars + 2 * kStages;
    uint64_t* acc_empty = acc_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEM);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);

    const int warp = threadIdx.x / 32;
    const uint32_t lane = lane_id();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], kEpiWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmap_o);
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_v);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    griddep_wait();                 // o may be the previous kernel's output until here

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
                const int h = u % kH;
                const int m0 = (u / kH) * kBM;
                for (int kb = 0; kb < kKB; ++kb, ++it) {
                    const int st = it % kStages;
                    if (!(ok = mbar_wait_spin(&empty[st], ((it / kStages) & 1) ^ 1, abort_flag, p.status))) break;
                    mbar_arrive_expect_tx(&full[st], kABytes + kBBytes);
                    // rows m0.. of head h's latent slice (rows past R arrive as zeros)
                    tma_load_2d(sA + st * kABytes, &tmap_o, &full[st], h * kDv + kb * 64, m0);
                    // the head's 256 feature rows, dims kb*64 ..
                    tma_load_2d(sB + st * kBBytes, &tmap_w, &full[st], kb * 64, h * kE);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int it = 0, ui = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x, ++ui) {
                const int acc = ui & 1;
                if (!(ok = mbar_wait_spin(&acc_empty[acc], ((ui >> 1) & 1) ^ 1, abort_flag, p.status))) break;
                tc_fence_after();
                const uint32_t d = tmem_base + acc * kE;
                for (int kb = 0; kb < kKB; ++kb, ++it) {
                    const int st = it % kStages;
                    if (!(ok = mbar_wait_spin(&full[st], (it / kStages) & 1, abort_flag, p.status))) break;
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(sA + st * kABytes);
                    const uint32_t b_base = smem_u32(sB + st * kBBytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = sdesc_sw128(a_base + kk * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(b_base + kk * 32, 16, 1024);
                        mma_bf16_ss(d, ad, bd, IDESC, (kb | kk) != 0);
                    }
                    mma_commit(&empty[st]);
                }
                if (ok) mma_commit(&acc_full[acc]);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 2..9)
        const int e = warp - 2;                         // 0..7
        const int quad = warp & 3;                      // TMEM lane quadrant of this warp
        const int half = e >> 2;                        // columns [128 half, 128 half + 128)
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        uint8_t* stg = smem + OFF_STG + e * kStgBytes;  // this warp's store box (1024-byte aligned)
        uint8_t* my_row = stg + lane * 128;             // row `lane` of the box
        int ui = 0;
        for (int u = blockIdx.x; u < p.n_units; u += gridDim.x, ++ui) {
            const int h = u % kH;
            const int row0 = (u / kH) * kBM + quad * 32;   // first row of this warp's 32
            const int acc = ui & 1;
            // warp-uniform outcome: the TMEM loads below are warp-collective
            if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[acc], (ui >> 1) & 1, abort_flag, p.status))) break;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t x[32];
                tmem_ld32(tmem_base + lane_addr + acc * kE + half * 128 + c * 32, x);
                tmem_ld_wait();
                if (c == 3) {   // every TMEM read of this accumulator is done
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&acc_empty[acc]);
                }
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1]));
                if ((c & 1) == 0) {   // the box is about to be refilled: its previous store has read it
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
                }
                // 16-byte chunks 4 (c & 1) .. + 3 of the 128-byte row, 128-byte swizzle
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int chunk = 4 * (c & 1) + i;
                    *reinterpret_cast<uint4*>(my_row + ((chunk ^ (int)(lane & 7)) << 4)) =
                        make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
                if (c & 1) {   // 64 columns complete: one TMA store of the 32 x 64 box
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmap_v, stg, h * kE + half * 128 + (c >> 1) * 64, row0);
                        bulk_commit();
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace

dsa_status_t launch_value_up_proj(const void* o, const void* wv_b, int R, void* v, cudaStream_t stream) {
    CUtensorMap to, tw;
    dsa_status_t st;
    // o as R rows of 64 * 512 elements; a box is 64 dims of one head for 128 rows
    if ((st = make_tmap_bf16_2d(&to, o, (uint64_t)kH * kDv, (uint64_t)R, (uint64_t)kH * kDv * 2, 64, kBM)) != DSA_OK)
        return st;
    // wv_b as 64 * 256 feature rows of 512 dims; a box is one head's 256 rows x 64 dims
    if ((st = make_tmap_bf16_2d(&tw, wv_b, kDv, (uint64_t)kH * kE, kDv * 2, 64, kE)) != DSA_OK) return st;
    // v as R rows of 64 * 256 elements; a store box is 64 features of one head for 32 rows
    CUtensorMap tv;
    if ((st = make_tmap_bf16_2d(&tv, v, (uint64_t)kH * kE, (uint64_t)R, (uint64_t)kH * kE * 2, 64, 32)) != DSA_OK)
        return st;
    if ((st = ensure_smem_attr(reinterpret_cast<const void*>(value_up_proj_kernel), SMEM_BYTES)) != DSA_OK)
        return st;
    VprojParams p;
    p.R = R;
    const long long units = (long long)kH * ceil_div(R, kBM);
    if (units > 0x7FFFFFFFLL) return DSA_ERR_UNSUPPORTED_SHAPE;
    p.n_units = (int)units;
    p.status = device_status_ptr();
    const int grid = p.n_units < device_sm_count() ? p.n_units : device_sm_count();
    if (launch_pdl(value_up_proj_kernel, dim3(grid), dim3(kThreads), SMEM_BYTES, stream, to, tw, tv, p) != cudaSuccess)
        return DSA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
