// dsa_internal.h -- host-side helpers shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <utility>

#include "../../include/dsa.h"

namespace dsa {

// Number of SMs of the current device (cached per device).
int device_sm_count();
size_t device_l2_bytes();   // L2 size of the current device (0 if unknown)
// DSA_OK when the current device is compute capability 10.3.
dsa_status_t check_device();
// Device address of the sticky error word on the current device (nullptr if
// it cannot be obtained; kernels then skip the report).
int32_t* device_status_ptr();
// Raise the dynamic shared-memory limit of `func` on the current device once.
dsa_status_t ensure_smem_attr(const void* func, int bytes);

// 2D bf16 tensor map: `rows` rows of `cols` elements (row pitch `row_bytes`),
// box = box_cols x box_rows, 128-byte swizzle, zero fill out of bounds.
dsa_status_t make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                               uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows);

// Launch with programmatic dependent launch allowed: the launch is prepared
// while the previous kernel on the stream runs and the kernel starts as that
// kernel's CTAs exit; every kernel of the library runs its prologue (barriers,
// TMEM allocation) and then waits for its predecessor (griddepcontrol.wait)
// before it touches global memory.  No kernel triggers its successor early:
// measured on GB300, successor CTAs waiting next to running ones slowed the
// batch-8 decode step (36.8 vs 28.7 us as a graph).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Page table of a paged key cache: logical key j of sequence b is pool row
// table[b * stride + (j >> shift)] * 2^shift + (j & (2^shift - 1)).  A null
// table means the dense layout, row b * Nmax + j.
struct PageTable {
    const int32_t* table;
    int stride;      // entries per sequence
    int shift;       // log2(page_size)
    int num_pages;   // pages in the pool
};

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Launch entry points implemented in the kernel files.
dsa_status_t launch_indexer(const void* q_idx, const void* k_idx, const float* w, const int32_t* q_pos0,
                            const int32_t* kv_len, int B, int L, int Nmax, float* scores, int64_t ld,
                            const PageTable& pages, cudaStream_t stream);
dsa_status_t launch_topk(const float* scores, int64_t ld, const int32_t* q_pos0, const int32_t* kv_len, int B,
                         int L, int Nmax, int top_k, int32_t* idx, cudaStream_t stream);
dsa_status_t launch_attn_prefill(const void* q, const void* kv, const int32_t* idx, int L, int N, int top_k,
                                 float scale, void* out, int out_f32, float* lse, const PageTable& pages,
                                 cudaStream_t stream);
size_t attn_decode_workspace(int B, int top_k);
dsa_status_t launch_attn_decode_noalloc(const void* q, const void* kv, const int32_t* kv_len, const int32_t* idx,
                                        int B, int Nmax, int top_k, float scale, void* out, int out_f32,
                                        float* lse, cudaStream_t stream);
dsa_status_t launch_attn_decode(const void* q, const void* kv, const int32_t* kv_len, const int32_t* idx, int B,
                                int Nmax, int top_k, float scale, void* out, int out_f32, float* lse,
                                void* workspace, const PageTable& pages, cudaStream_t stream);
dsa_status_t launch_value_up_proj(const void* o, const void* wv_b, int R, void* v, cudaStream_t stream);

}  // namespace dsa
