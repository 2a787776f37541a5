// api.cu -- the C ABI declared in include/dsa.h: argument validation (all on
// the host, before any launch), status codes, device checks, TMA descriptor
// encoding and the sticky device error word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "dsa_internal.h"
#include "dsa_ptx.cuh"

namespace dsa {

__device__ int32_t g_dev_status = 0;

namespace {
std::atomic<int32_t*> g_status_ptr[64];
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_l2_bytes[kMaxDevices];
std::atomic<int> g_cc_ok[kMaxDevices];  // 0 unknown, 1 ok, 2 not sm_103
std::mutex g_attr_mu;

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}
}  // namespace

int32_t* device_status_ptr() {
    int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    int32_t* ptr = g_status_ptr[dev].load();
    if (!ptr) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, g_dev_status) != cudaSuccess) return nullptr;
        ptr = static_cast<int32_t*>(a);
        g_status_ptr[dev].store(ptr);
    }
    return ptr;
}

int device_sm_count() {
    int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 148;
    int v = g_sm_count[dev].load();
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        g_sm_count[dev].store(v);
    }
    return v;
}

size_t device_l2_bytes() {
    int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 0;
    int v = g_l2_bytes[dev].load();
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess || v <= 0) v = 0;
        g_l2_bytes[dev].store(v);
    }
    return (size_t)v;
}

dsa_status_t check_device() {
    int dev = current_device();
    if (dev < 0) return DSA_ERR_CUDA;
    if (dev >= kMaxDevices) return DSA_ERR_UNSUPPORTED_DEVICE;
    int s = g_cc_ok[dev].load();
    if (s == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return DSA_ERR_CUDA;
        s = (major == 10 && minor == 3) ? 1 : 2;
        g_cc_ok[dev].store(s);
    }
    return s == 1 ? DSA_OK : DSA_ERR_UNSUPPORTED_DEVICE;
}

dsa_status_t ensure_smem_attr(const void* func, int bytes) {
    // cheap enough to repeat; serialised so concurrent first calls do not race
    std::lock_guard<std::mutex> g(g_attr_mu);
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return DSA_ERR_CUDA;
    return DSA_OK;
}

namespace {
dsa_status_t make_tmap_impl(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint64_t row_bytes,
                            uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz) {
    auto fn = encode_fn();
    if (!fn) return DSA_ERR_CUDA;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DSA_OK : DSA_ERR_CUDA;
}
}  // namespace

dsa_status_t make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint64_t row_bytes,
                               uint32_t box_cols, uint32_t box_rows) {
    return make_tmap_impl(map, base, cols, rows, row_bytes, box_cols, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace dsa

using namespace dsa;

namespace selftest {
// One thread waits, with the kernels' bounded wait routine, for phase 0 of a fresh mbarrier that
// nothing arrives on: the wait gives up after limit_ns and records the timeout in the status word.
__global__ void wait_timeout_selftest_kernel(int32_t* status, uint64_t limit_ns, int spin) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    volatile int* abort_ptr = &abort_flag;
    if (spin)
        (void)mbar_wait_spin(&bar, 0, abort_ptr, status, limit_ns);
    else
        (void)mbar_wait(&bar, 0, abort_ptr, status, limit_ns);
}
}  // namespace selftest

extern "C" {

const char* dsa_status_string(dsa_status_t s) {
    switch (s) {
        case DSA_OK: return "ok";
        case DSA_ERR_INVALID_ARG: return "invalid argument (null pointer, non-positive size or bad stride)";
        case DSA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (fixed head counts/widths, 1 <= top_k <= 2048)";
        case DSA_ERR_MISALIGNED: return "pointer or row stride not 16-byte aligned";
        case DSA_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than the *_workspace_size() query";
        case DSA_ERR_CUDA: return "CUDA runtime call or kernel launch failed";
        case DSA_ERR_DEVICE_TIMEOUT: return "an in-kernel wait ran past its limit";
        case DSA_ERR_DEVICE_BOUNDS: return "a selected key index was outside the cache (access skipped)";
        case DSA_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3 (sm_103a)";
        case DSA_ERR_SCRATCH_TOO_SMALL:
            return "request exceeds the fixed device scratch of mla_sparse_attn_decode_noalloc (B <= 63)";
        default: return "unknown status";
    }
}

int dsa_abi_version(void) { return DSA_ABI_VERSION; }

dsa_status_t dsa_indexer_scores(const void* q_idx, const void* k_idx, const float* w, const int32_t* q_pos0,
                                const int32_t* kv_len, int B, int L, int Nmax, float* scores, int64_t ld,
                                void* stream) {
    if (!q_idx || !k_idx || !w || !q_pos0 || !kv_len || !scores) return DSA_ERR_INVALID_ARG;
    if (B < 1 || L < 1 || Nmax < 1 || ld < Nmax) return DSA_ERR_INVALID_ARG;
    if ((long long)B * L * DSA_INDEXER_HEADS > 0x7FFFFFFFLL || (long long)B * Nmax > 0x7FFFFFFFLL)
        return DSA_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(w) || !aligned16(scores) || (ld % 4) != 0)
        return DSA_ERR_MISALIGNED;
    dsa_status_t st = check_device();
    if (st != DSA_OK) return st;
    return launch_indexer(q_idx, k_idx, w, q_pos0, kv_len, B, L, Nmax, scores, ld, PageTable{},
                          static_cast<cudaStream_t>(stream));
}

namespace {
// Host checks of a page table's geometry; fills `pt` on success.
dsa_status_t make_page_table(const int32_t* table, int stride, int page_size, int num_pages, int Nmax,
                             PageTable* pt) {
    if (!table) return DSA_ERR_INVALID_ARG;
    if (stride < 1 || num_pages < 1) return DSA_ERR_INVALID_ARG;
    if (page_size < 16 || page_size > 65536 || (page_size & (page_size - 1)) != 0) return DSA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)num_pages * page_size > 0x7FFFFFFFLL) return DSA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)stride * page_size < Nmax) return DSA_ERR_INVALID_ARG;
    int shift = 0;
    while ((1 << shift) < page_size) ++shift;
    *pt = PageTable{table, stride, shift, num_pages};
    return DSA_OK;
}
}  // namespace

dsa_status_t dsa_indexer_scores_paged(const void* q_idx, const void* k_pool, const float* w, const int32_t* q_pos0,
                                      const int32_t* kv_len, const int32_t* block_table, int bt_stride,
                                      int page_size, int num_pages, int B, int L, int Nmax, float* scores,
                                      int64_t ld, void* stream) {
    if (!q_idx || !k_pool || !w || !q_pos0 || !kv_len || !scores) return DSA_ERR_INVALID_ARG;
    if (B < 1 || L < 1 || Nmax < 1 || ld < Nmax) return DSA_ERR_INVALID_ARG;
    if ((long long)B * L * DSA_INDEXER_HEADS > 0x7FFFFFFFLL) return DSA_ERR_UNSUPPORTED_SHAPE;
    PageTable pt;
    dsa_status_t st = make_page_table(block_table, bt_stride, page_size, num_pages, Nmax, &pt);
    if (st != DSA_OK) return st;
    if ((long long)B * bt_stride > 0x7FFFFFFFLL) return DSA_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(q_idx) || !aligned16(k_pool) || !aligned16(w) || !aligned16(scores) || (ld % 4) != 0)
        return DSA_ERR_MISALIGNED;
    if ((st = check_device()) != DSA_OK) return st;
    return launch_indexer(q_idx, k_pool, w, q_pos0, kv_len, B, L, Nmax, scores, ld, pt,
                          static_cast<cudaStream_t>(stream));
}

size_t dsa_topk_workspace_size(int B, int L, int Nmax, int top_k) {
    (void)B;
    (void)L;
    (void)Nmax;
    (void)top_k;
    return 0;
}

dsa_status_t dsa_topk(const float* scores, int64_t ld, const int32_t* q_pos0, const int32_t* kv_len, int B, int L,
                      int Nmax, int top_k, int32_t* idx, void* workspace, size_t ws_bytes, void* stream) {
    (void)workspace;
    (void)ws_bytes;
    if (!scores || !q_pos0 || !kv_len || !idx) return DSA_ERR_INVALID_ARG;
    if (B < 1 || L < 1 || Nmax < 1 || ld < Nmax) return DSA_ERR_INVALID_ARG;
    if (top_k < 1 || top_k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)B * L > 0x7FFFFFFFLL) return DSA_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(scores) || (ld % 4) != 0) return DSA_ERR_MISALIGNED;
    dsa_status_t st = check_device();
    if (st != DSA_OK) return st;
    return launch_topk(scores, ld, q_pos0, kv_len, B, L, Nmax, top_k, idx, static_cast<cudaStream_t>(stream));
}

size_t mla_sparse_attn_workspace_size(int B, int L, int top_k, int is_decode) {
    (void)L;
    if (!is_decode || B < 1 || top_k < 1) return 0;
    return attn_decode_workspace(B, top_k);
}

dsa_status_t mla_sparse_attn_prefill(const void* q, const void* kv, const int32_t* idx, int L, int N, int top_k,
                                     float scale, void* out, int out_dtype, float* lse, void* workspace,
                                     size_t ws_bytes, void* stream) {
    (void)workspace;
    (void)ws_bytes;
    if (!q || !kv || !idx || !out) return DSA_ERR_INVALID_ARG;
    if (out_dtype != DSA_OUT_F32 && out_dtype != DSA_OUT_BF16) return DSA_ERR_INVALID_ARG;
    if (L < 1 || N < 1) return DSA_ERR_INVALID_ARG;
    if (top_k < 1 || top_k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)L * DSA_HEADS > 0x7FFFFFFFLL) return DSA_ERR_UNSUPPORTED_SHAPE;
    if (!(scale > 0.f) || !(scale < 1e30f)) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kv) || !aligned16(out)) return DSA_ERR_MISALIGNED;
    dsa_status_t st = check_device();
    if (st != DSA_OK) return st;
    return launch_attn_prefill(q, kv, idx, L, N, top_k, scale, out, out_dtype == DSA_OUT_F32, lse, PageTable{},
                               static_cast<cudaStream_t>(stream));
}

dsa_status_t mla_sparse_attn_prefill_paged(const void* q, const void* kv_pool, const int32_t* block_table,
                                           int page_size, int num_pages, const int32_t* idx, int L, int N,
                                           int top_k, float scale, void* out, int out_dtype, float* lse,
                                           void* workspace, size_t ws_bytes, void* stream) {
    (void)workspace;
    (void)ws_bytes;
    if (!q || !kv_pool || !idx || !out) return DSA_ERR_INVALID_ARG;
    if (out_dtype != DSA_OUT_F32 && out_dtype != DSA_OUT_BF16) return DSA_ERR_INVALID_ARG;
    if (L < 1 || N < 1) return DSA_ERR_INVALID_ARG;
    if (top_k < 1 || top_k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED_SHAPE;
    if ((long long)L * DSA_HEADS > 0x7FFFFFFFLL) return DSA_ERR_UNSUPPORTED_SHAPE;
    if (!(scale > 0.f) || !(scale < 1e30f)) return DSA_ERR_INVALID_ARG;
    PageTable pt;
    // one sequence: its table row holds ceil(N / page_size) entries
    const int stride = page_size > 0 ? (int)(((long long)N + page_size - 1) / page_size) : 0;
    dsa_status_t st = make_page_table(block_table, stride, page_size, num_pages, N, &pt);
    if (st != DSA_OK) return st;
    if (!aligned16(q) || !aligned16(kv_pool) || !aligned16(out)) return DSA_ERR_MISALIGNED;
    if ((st = check_device()) != DSA_OK) return st;
    return launch_attn_prefill(q, kv_pool, idx, L, N, top_k, scale, out, out_dtype == DSA_OUT_F32, lse, pt,
                               static_cast<cudaStream_t>(stream));
}

dsa_status_t mla_sparse_attn_decode(const void* q, const void* kv, const int32_t* kv_len, const int32_t* idx, int B,
                                    int Nmax, int top_k, float scale, void* out, int out_dtype, float* lse,
                                    void* workspace, size_t ws_bytes, void* stream) {
    if (!q || !kv || !kv_len || !idx || !out || !workspace) return DSA_ERR_INVALID_ARG;
    if (out_dtype != DSA_OUT_F32 && out_dtype != DSA_OUT_BF16) return DSA_ERR_INVALID_ARG;
    if (B < 1 || Nmax < 1) return DSA_ERR_INVALID_ARG;
    if (top_k < 1 || top_k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED_SHAPE;
    if (!(scale > 0.f) || !(scale < 1e30f)) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kv) || !aligned16(out) || !aligned16(workspace)) return DSA_ERR_MISALIGNED;
    if (ws_bytes < attn_decode_workspace(B, top_k)) return DSA_ERR_WORKSPACE_TOO_SMALL;
    dsa_status_t st = check_device();
    if (st != DSA_OK) return st;
    return launch_attn_decode(q, kv, kv_len, idx, B, Nmax, top_k, scale, out, out_dtype == DSA_OUT_F32, lse,
                              workspace, PageTable{}, static_cast<cudaStream_t>(stream));
}

dsa_status_t mla_sparse_attn_decode_paged(const void* q, const void* kv_pool, const int32_t* kv_len,
                                          const int32_t* block_table, int bt_stride, int page_size, int num_pages,
                                          const int32_t* idx, int B, int Nmax, int top_k, float scale, void* out,
                                          int out_dtype, float* lse, void* workspace, size_t ws_bytes,
                                          void* stream) {
    if (!q || !kv_pool || !kv_len || !idx || !out || !workspace) return DSA_ERR_INVALID_ARG;
    if (out_dtype != DSA_OUT_F32 && out_dtype != DSA_OUT_BF16) return DSA_ERR_INVALID_ARG;
    if (B < 1 || Nmax < 1) return DSA_ERR_INVALID_ARG;
    if (top_k < 1 || top_k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED_SHAPE;
    if (!(scale > 0.f) || !(scale < 1e30f)) return DSA_ERR_INVALID_ARG;
    PageTable pt;
    dsa_status_t st = make_page_table(block_table, bt_stride, page_size, num_pages, Nmax, &pt);
    if (st != DSA_OK) return st;
    if ((long long)B * bt_stride > 0x7FFFFFFFLL) return DSA_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(q) || !aligned16(kv_pool) || !aligned16(out) || !aligned16(workspace)) return DSA_ERR_MISALIGNED;
    if (ws_bytes < attn_decode_workspace(B, top_k)) return DSA_ERR_WORKSPACE_TOO_SMALL;
    if ((st = check_device()) != DSA_OK) return st;
    return launch_attn_decode(q, kv_pool, kv_len, idx, B, Nmax, top_k, scale, out, out_dtype == DSA_OUT_F32, lse,
                              workspace, pt, static_cast<cudaStream_t>(stream));
}

dsa_status_t mla_sparse_attn_decode_noalloc(const void* q, const void* kv, const int32_t* kv_len,
                                            const int32_t* idx, int B, int Nmax, int top_k, float scale, void* out,
                                            int out_dtype, float* lse, void* stream) {
    if (!q || !kv || !kv_len || !idx || !out) return DSA_ERR_INVALID_ARG;
    if (out_dtype != DSA_OUT_F32 && out_dtype != DSA_OUT_BF16) return DSA_ERR_INVALID_ARG;
    if (B < 1 || Nmax < 1) return DSA_ERR_INVALID_ARG;
    if (top_k < 1 || top_k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED_SHAPE;
    if (!(scale > 0.f) || !(scale < 1e30f)) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kv) || !aligned16(out)) return DSA_ERR_MISALIGNED;
    if (B > DSA_NOALLOC_MAX_BATCH) return DSA_ERR_SCRATCH_TOO_SMALL;
    dsa_status_t st = check_device();
    if (st != DSA_OK) return st;
    return launch_attn_decode_noalloc(q, kv, kv_len, idx, B, Nmax, top_k, scale, out, out_dtype == DSA_OUT_F32,
                                      lse, static_cast<cudaStream_t>(stream));
}

dsa_status_t mla_value_up_proj(const void* o, const void* wv_b, int R, void* v, void* stream) {
    if (!o || !wv_b || !v) return DSA_ERR_INVALID_ARG;
    if (R < 1) return DSA_ERR_INVALID_ARG;
    if ((long long)R * DSA_HEADS > 0x7FFFFFFFLL) return DSA_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(o) || !aligned16(wv_b) || !aligned16(v)) return DSA_ERR_MISALIGNED;
    dsa_status_t st = check_device();
    if (st != DSA_OK) return st;
    return launch_value_up_proj(o, wv_b, R, v, static_cast<cudaStream_t>(stream));
}

int dsa_indexer_source_layer(int layer, int topk_freq, int skip_offset) {
    if (layer < 0 || topk_freq < 1 || skip_offset < 1) return -1;
    if (layer < skip_offset) return layer;
    // layers skip_offset + topk_freq - 1, + 2 topk_freq - 1, ... run the indexer
    const int k = (int)(((long long)layer - skip_offset + 1) % topk_freq);
    return layer - k;
}

dsa_status_t dsa_selftest_wait_timeout(int spin, uint64_t limit_ns, void* stream) {
    if (spin != 0 && spin != 1) return DSA_ERR_INVALID_ARG;
    if (limit_ns == 0 || limit_ns > 1000000000ull) return DSA_ERR_INVALID_ARG;
    dsa_status_t st = check_device();
    if (st != DSA_OK) return st;
    selftest::wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(device_status_ptr(), limit_ns, spin);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

dsa_status_t dsa_device_status(void* stream, int32_t* code_out, int reset) {
    if (!code_out) return DSA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return DSA_ERR_CUDA;
    int32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, g_dev_status, sizeof v) != cudaSuccess) return DSA_ERR_CUDA;
    if (reset) {
        int32_t z = 0;
        if (cudaMemcpyToSymbol(g_dev_status, &z, sizeof z) != cudaSuccess) return DSA_ERR_CUDA;
    }
    *code_out = (v & DEV_ERR_TIMEOUT) ? DSA_ERR_DEVICE_TIMEOUT : (v & DEV_ERR_BOUNDS) ? DSA_ERR_DEVICE_BOUNDS : DSA_OK;
    return DSA_OK;
}

}  // extern "C"
