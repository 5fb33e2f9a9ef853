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
    float *fac;  // per-chunk factor cache written by the forward (L == 16), or NULL
    // backward only
    const float *dy, *dsT, *ckpt_in;
    const float *fac_in;  // factor cache from the forward, or NULL (recomputed)
    float *dr, *dw, *dk, *dv, *da, *db, *ds0;
    unsigned *err;  // device flag a kernel sets when a bounded wait on its copies times out
    // 1: the inputs w, a, b hold the producers' inputs w_pre, kk, avec (w = exp(-0.606531
    // sigmoid(w_pre)), a = -kk, b = kk * avec) and the backward writes the gradients of
    // those (dw_pre, dkk, davec) into dw, da, db
    int prod;
    // GroupNorm + bonus output epilogue (wkv7_forward_gn / wkv7_backward_gn), else NULL:
    // per-channel weights [H][64]; the forward's epilogue output o; the backward reads
    // the forward's y (y_in), takes do in dy, and writes per-(b,h) partial sums of
    // dgn_w, dgn_b, dr_k ([B*H][3][64]) into gn_part
    const float *gn_w, *gn_b, *r_k;
    float *o;
    const float *y_in;
    float *gn_part;
    // the state passes (the time split's segment summaries): 0 the whole call.
    // Forward: 1 only the end state sT (no y); 2 only the end state with v = 0
    // (the product of the transitions applied to s0; v and k are not read).
    // Backward: 1 only ds0 (r, w, a, b, dy and the factor cache are read).
    int state_only;
};

// Per-chunk factor cache: 2048 32-bit words per (b, h, 16-token chunk), in the
// register-fragment order of the backward's warps, so that both sides move it
// with 16-byte accesses over contiguous lanes.  Split operands are stored as
// bf16x2 (hi, lo) pairs of mma.m16n8k16 fragments; each 32-byte lane record
// is two 16-byte halves 512 bytes apart (half h of lane l at word 128 h + 4 l).
namespace fac {
constexpr int kWA = 0;      // W as an A fragment: halves {hi[0..3]}, {lo[0..3]}
constexpr int kMkA = 256;   // M_k' (= M_k W) as an A fragment, same packing
constexpr int kQB = 512;    // Q' as the B fragments of the two 8-column n-tiles: halves {b0.hi, b0.lo}, {b1.hi, b1.lo}
constexpr int kWQbB = 768;  // W Q_b, same packing
constexpr int kSA = 1024;   // SA fp32, 256 words per warp: halves = its two token tiles (4 accumulator values each)
constexpr int kWords = 2048;
}  // namespace fac

// Record an error for wkv7_last_error() and return `code` (C ABI layer).
int set_error(int code, const char *msg);
// The time split's segment passes: the chunked forward of B*T*H inputs from s0
// (NULL: zeros), writing only sT; state_only 1 reads w, k, v, a, b, state_only 2
// reads w, a, b (v = 0).  Arguments already checked by the caller.
int forward_state(int B, int T, int H, int dtype, const void *w, const void *k, const void *v, const void *a,
                  const void *b, const float *s0, float *sT, int state_only, cudaStream_t s);
// The state-gradient pass: ds0 of the chunked backward of B*T*H inputs (dsT
// NULL: zeros) from r, w, a, b, dy and the forward's factor cache, without
// the per-token gradients; bit-identical to the full backward's ds0.
// Arguments already checked by the caller.
int backward_state(int B, int T, int H, int dtype, const void *r, const void *w, const void *a, const void *b,
                   const float *factors, const float *dy, const float *dsT, float *ds0, cudaStream_t s);
// Host checks shared by every entry point, run before anything is launched:
// sizes and dtype, the required pointers (non-NULL when T > 0) and the
// optional ones (NULL allowed), 16-byte alignment of both, and an sm_103a
// current device.  Returns WKV7_OK or the error code, with the message set.
int check_call(int B, int T, int H, int N, int dtype, const void *const *req, const char *const *req_names, int nreq,
               const void *const *opt, const char *const *opt_names, int nopt);
// Device address of the current device's asynchronous-error flag (looked up
// once per device), or NULL with the error recorded.
unsigned *async_error_flag();

// Launchers (return the launch's cudaError_t).
cudaError_t launch_forward_plain(const SeqArgs &a, cudaStream_t s);
bool forward_chunk_supported(const SeqArgs &a);
cudaError_t launch_forward_chunk(const SeqArgs &a, cudaStream_t s);
cudaError_t launch_backward_plain(const SeqArgs &a, cudaStream_t s);
bool backward_chunk_supported(const SeqArgs &a);
cudaError_t launch_backward_chunk(const SeqArgs &a, cudaStream_t s);
cudaError_t launch_backward_state(const SeqArgs &a, cudaStream_t s);
bool backward_tc_supported(const SeqArgs &a);
cudaError_t launch_backward_tc(const SeqArgs &a, cudaStream_t s);
cudaError_t launch_gn_param_reduce(int B, int H, const float *part, float *dgn_w, float *dgn_b, float *dr_k,
                                   cudaStream_t s);
cudaError_t launch_decode_step(int B, int H, int dtype, const void *r, const void *w,
                               const void *k, const void *v, const void *a, const void *b,
                               float *state, float *y, cudaStream_t s);

}  // namespace wkv7
