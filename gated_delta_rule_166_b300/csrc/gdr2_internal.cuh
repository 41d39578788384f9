// Internal declarations shared by the libgdr2 translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdr2 {

// Element conversions for the two supported token dtypes.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Device-side failure codes written to the library's error word.
enum : int { kDevOk = 0, kDevTimeout = 1 };

struct ForwardArgs {
    const void *q, *k, *v, *b, *w, *g;
    const float* S0;
    void* o;
    float* ST;
    int64_t B, T, H, dk, dv;   // B sequences; T their common length when cu is null
    const int* cu;             // packed sequences: start offsets [B + 1] on the device, or null
    int64_t total;             // token rows of the packed tensors (cu != null)
    int in_dtype;        // GDR2_F32 / GDR2_BF16: q, k, v, b, w, log_decay
    int out_dtype;       // GDR2_F32 / GDR2_BF16: o
};

struct DecodeArgs {
    const void *q, *k, *v, *b, *w, *g;
    float* S;
    void* o;
    int64_t B, H, dk, dv;
    int in_dtype;
    int out_dtype;
};

// Launchers; each returns a gdr2_status value.  `err` is the device address
// of the library's error word (bounded waits record failures there).
int launch_recurrent(const ForwardArgs& a, cudaStream_t stream);
int launch_decode(const DecodeArgs& a, cudaStream_t stream);
int launch_chunked_bf16(const ForwardArgs& a, cudaStream_t stream, int* err);
bool chunked_bf16_supports(const ForwardArgs& a);

}  // namespace gdr2
