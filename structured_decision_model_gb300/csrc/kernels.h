// Host-side launchers of the head's kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

namespace clef {

// Kernels launched by the library since it was loaded.
extern std::atomic<uint64_t> g_kernel_launches;

// Counts a launch that the runtime accepted and passes the launch status on.
inline cudaError_t counted(cudaError_t e) {
    if (e == cudaSuccess) g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
    return e;
}

// Launch with programmatic stream serialization (see griddep_wait in common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return counted(cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...));
}

// ------------------------------------------------------------------ the GEMM

enum EpiKind : int {
    EPI_F32 = 0,        // out_f32 = acc + bias
    EPI_BF16 = 2,       // out_bf16 = act(acc + bias)
    EPI_KV_LNFOLD = 3,  // out_bf16 = rstd[m] * (acc - mu[m] * col_c[n]) + bias_f32[n], with mu and
                        // rstd the memory LayerNorm statistics of A's row m, computed in the kernel
};

struct GemmEpilogue {
    int kind = EPI_F32;
    int gelu = 0;
    const uint16_t* bias_bf16 = nullptr;  // [N]
    const float* bias_f32 = nullptr;      // [N]
    // LN fold: the row statistics are written to row_mu / row_rstd for rows m < M.  With
    // tile_rec given, row m belongs to record b = tile_rec[m / 128] and is a padding row
    // when m - rec_row_off[b] >= rec_len[b] (without: every row m < M is real); padding
    // rows get mu = rstd = 0 and are stored as zeros.  row_flags[g] (n_mtiles * 32 entries)
    // is set to `epoch` once rows 4g .. 4g + 3 are published.  The launcher gives each
    // launch a new epoch, so flags left by earlier launches never match; the caller clears
    // the flags beforehand so that no other earlier content can match either.
    float* row_mu = nullptr;              // [M] out (LN fold)
    float* row_rstd = nullptr;            // [M] out (LN fold)
    const int32_t* tile_rec = nullptr;    // [n_mtiles] record of each 128-row tile (LN fold)
    const int32_t* rec_row_off = nullptr; // [records] first row of each record (LN fold)
    const int32_t* rec_len = nullptr;     // [records] real rows of each record (LN fold)
    uint64_t* row_flags = nullptr;        // [n_mtiles * 32] (LN fold)
    uint64_t epoch = 0;                   // set by launch_gemm
    const float* col_c = nullptr;         // [N]    (LN fold)
    void* out = nullptr;
    int64_t ldo = 0;
    int M = 0;  // rows that are stored (m < M)
};

struct GemmProblem {
    const uint16_t* A = nullptr;  // bf16 [a_rows, K], row stride lda
    int64_t lda = 0;
    int64_t a_rows = 0;           // rows addressable through A's tensor map
    const uint16_t* B = nullptr;  // bf16 [N, K], row stride ldb
    int64_t ldb = 0;
    int N = 0, K = 0;
    int n_mtiles = 0;                        // 128-row output tiles
    const int32_t* a_row_of_mtile = nullptr; // device [n_mtiles]: first A row of each tile (null: 128 * tile)
    // split K across a thread-block cluster when the output tiles cannot fill the GPU
    // (needs no scratch: the partial tiles are summed in distributed shared memory)
    bool allow_split = false;
    // B is never written by a kernel that may still be running on the stream (weights): its
    // first tiles may then be requested before waiting for the previous kernel of the stream
    bool b_is_weight = false;
    // deferred split-K (defer_splits > 0, widths from partial_split_config): defer_splits
    // CTAs per output tile of width defer_bn, each storing its raw fp32 partial product into
    // slab sp of the epilogue output (slab stride part_stride elements; the epilogue must be
    // a plain EPI_F32 store); the consumer sums the slabs in split order
    int defer_splits = 0;
    int defer_bn = 0;
    int64_t part_stride = 0;
};

int num_sms();

// Tile width and split count of a deferred split-K product: a function of the
// output-tile count, N and K only.
void partial_split_config(int n_mtiles, int N, int K, int* bn, int* splits);

// 2-D TMA descriptor of a row-major bf16 matrix [rows][inner] (row stride in elements),
// 64-element x box_rows box, 128-byte swizzle.  Returns false if the driver rejects it.
bool make_tma_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride_elems,
                      uint32_t box_rows);
cudaError_t launch_gemm(const GemmProblem& p, const GemmEpilogue& e, int* dev_flags, cudaStream_t s,
                        int force_bn = 0);

}  // namespace clef
