// sd_host.h -- host-side helpers shared by the libsdgqa entry points (not installed).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdarg>
#include <cstdio>
#include <utility>

#include "../../include/sd.h"

namespace sd {

// Records the detail of a failed call for sd_last_error_message() (thread-local).
void set_error(const char* fmt, ...);
void clear_error();

// Number of SMs of the current device (queried once per device, then cached).
int num_sms();

// Maximum opt-in dynamic shared memory per block of the current device (cached).
int max_smem_optin();

// Host-side checks of an sd_attend_args shared by the calls that take one; `who` names the
// call in the error message.
sd_status validate_attend_args(const sd_attend_args* a, const char* who);

// Top-k of few long rows by thread-block clusters (the selection of sd_select_attend alone):
// false when the rows need clusters of one CTA (nothing launched), else launches and sets
// *status.
bool topk_by_clusters(const float* scores, int rows, int N, int k, int32_t* idx, uint32_t* key_hist,
                      cudaStream_t st, sd_status* status);

// sd_decode_step's path for block selection over short score rows (one thread-block cluster
// per KV group): whether a validated request takes it, and its launch.
bool block_step_eligible(const sd_decode_step_args* a);
sd_status block_step_launch(const sd_decode_step_args* a, cudaStream_t st);
// sd_gather_attend's tiled path over a cache in HBM, dense or blocks of 16 or more rows
// (dense_attend.cu): whether it applies,
// and its launch, at most max_splits splits (partials in ws_o/ws_m/ws_l with RP rows per
// split when more than one; *splits_used tells how many).
bool dense_tma_eligible(const sd_attend_args* a);
int dense_tma_ctas_per_sm(const sd_attend_args* a);
int dense_tma_max_split_rows();  // list rows a split of a block-sparse call may hold
sd_status dense_tma_launch(const sd_attend_args* a, int max_splits, int RP, float* ws_o, float* ws_m, float* ws_l,
                           int* splits_used, cudaStream_t st);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Device address of pinned, mapped host memory (NULL if h is not such memory).
inline const uint8_t* mapped_host_ptr(const void* h) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, h) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return nullptr;
    return static_cast<const uint8_t*>(at.devicePointer);
}

inline bool valid_dtype(int dt) { return dt == SD_F32 || dt == SD_BF16; }
inline int dtype_bytes(int dt) { return dt == SD_F32 ? 4 : 2; }  // F32 4, BF16 and F16 2

// Maps the last launch error to a status (and records it).
inline sd_status launch_status(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("%s: launch failed: %s", what, cudaGetErrorString(e));
        return SD_ERR_CUDA;
    }
    return SD_OK;
}

// 2-D tensor map of 16-bit elements (bf16, or fp16 with f16) over [nrows, d] (row-major),
// box = 64 columns x box_rows rows, 128-byte swizzle, zero fill outside the tensor; false
// when the driver's encoder is unavailable or rejects the map.
bool make_tensor_map_2d(CUtensorMap* m, const void* base, uint64_t nrows, int d, int box_rows, bool f16);

// The indexer on the tensor cores (index_score_tc.cu): bf16 keys and queries, or fp16 ones
// (f16).
sd_status index_score_tc_launch(const void* q_idx, const void* k_idx, int rows, int V, int N, int d_idx,
                                float* scores, uint32_t* key_hist, int32_t* err_word, int per_query, bool f16, cudaStream_t st);

// Launches `kern` as a programmatic dependent of the preceding kernel in the stream: it
// may be scheduled before that kernel finishes and must call pdl_wait() before reading
// anything the preceding work wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace sd

#define SD_REQUIRE(cond, ...)                 \
    do {                                      \
        if (!(cond)) {                        \
            ::sd::set_error(__VA_ARGS__);     \
            return SD_ERR_INVALID_ARG;        \
        }                                     \
    } while (0)

#define SD_CUDA_CHECK(call, what)                                                     \
    do {                                                                              \
        cudaError_t e_ = (call);                                                      \
        if (e_ != cudaSuccess) {                                                      \
            ::sd::set_error("%s: %s", what, cudaGetErrorString(e_));                  \
            return SD_ERR_CUDA;                                                       \
        }                                                                             \
    } while (0)
