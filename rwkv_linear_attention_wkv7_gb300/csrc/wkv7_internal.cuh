// Internal declarations shared by the WKV7 CUDA translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace wkv7 {

constexpr int kN = 64;  // head size

// Pointers of one call, already validated by the C ABI layer.
struct SeqArgs {
    int B, T, H, L, nck;
    int dtype;  // 0 = fp32, 1 = bf16
    const void *r, *w, *k, *v, *a, *b;
    const float *s0;
    float *y, *sT, *ckpt;
    // backward only
    const float *dy, *dsT, *ckpt_in;
    float *dr, *dw, *dk, *dv, *da, *db, *ds0;
};

// Launchers (return the launch's cudaError_t).
cudaError_t launch_forward_plain(const SeqArgs &a, cudaStream_t s);
bool forward_chunk_supported(const SeqArgs &a);
cudaError_t launch_forward_chunk(const SeqArgs &a, cudaStream_t s);
cudaError_t launch_backward_plain(const SeqArgs &a, cudaStream_t s);
bool backward_chunk_supported(const SeqArgs &a);
cudaError_t launch_backward_chunk(const SeqArgs &a, cudaStream_t s);
cudaError_t launch_decode_step(int B, int H, int dtype, const void *r, const void *w,
                               const void *k, const void *v, const void *a, const void *b,
                               float *state, float *y, cudaStream_t s);

}  // namespace wkv7
