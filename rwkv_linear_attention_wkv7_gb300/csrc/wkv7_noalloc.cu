// wkv7_forward_backward_noalloc: forward + backward with the per-chunk factor
// cache held in a fixed-size array inside the library, for callers that can
// allocate no device memory (the declaration in wkv7.h says who and why).
#include <cstdio>
#include <mutex>

#include "wkv7.h"
#include "wkv7_internal.cuh"

namespace {

constexpr long long kMaxChunkHeads = WKV7_NOALLOC_MAX_CHUNK_HEADS;
constexpr long long kScratchFloats = kMaxChunkHeads * wkv7::fac::kWords;  // 32 MiB

// The factor cache of every call on this device.  In host code this name is
// only a stand-in for the symbol; kernels get the device address looked up
// below.
static __device__ __align__(256) float g_factor_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_factor_scratch on the current device, looked up once
// per device with that device current.
int scratch_address(float **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return wkv7::set_error(WKV7_EUNSUPPORTED, "no CUDA device available");
    }
    if (dev < 0 || dev >= kMaxDevices)
        return wkv7::set_error(WKV7_EUNSUPPORTED, "device index beyond the no-alloc entry point's table");
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return wkv7::set_error(WKV7_EUNSUPPORTED, "cannot query the current device");
    }
    if (major != 10 || minor != 3) return wkv7::set_error(WKV7_EUNSUPPORTED, "this library is built for sm_103a only");
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_factor_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            char msg[200];
            snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the factor scratch failed: %s", cudaGetErrorString(e));
            return wkv7::set_error(WKV7_ECUDA, msg);
        }
        g_scratch_ptr[dev] = static_cast<float *>(p);
    }
    *out = g_scratch_ptr[dev];
    return WKV7_OK;
}

}  // namespace

extern "C" int wkv7_forward_backward_noalloc(int B, int T, int H, int N, wkv7_dtype dtype, const void *r,
                                             const void *w, const void *k, const void *v, const void *a,
                                             const void *b, const float *s0, const float *dy, const float *dsT,
                                             float *y, float *sT, float *ckpt, float *dr, float *dw, float *dk,
                                             float *dv, float *da, float *db, float *ds0, void *stream) {
    if (B < 1 || H < 1 || T < 0)
        return wkv7::set_error(WKV7_EINVAL, "B and H must be >= 1 and T >= 0");
    if (T > 0 && !ckpt) return wkv7::set_error(WKV7_EINVAL, "ckpt is NULL (the backward half reads it)");
    const long long chunk_heads = (long long)B * H * (((long long)T + 15) / 16);
    if (chunk_heads > kMaxChunkHeads) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "B*H*ceil(T/16) = %lld exceeds the no-alloc factor scratch of %lld chunk-heads (32 MiB)",
                 chunk_heads, kMaxChunkHeads);
        return wkv7::set_error(WKV7_EINVAL, msg);
    }
    float *scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc != WKV7_OK) return rc;
    rc = wkv7_forward(B, T, H, N, dtype, r, w, k, v, a, b, s0, y, sT, ckpt, scratch, 16, stream);
    if (rc != WKV7_OK) return rc;
    return wkv7_backward(B, T, H, N, dtype, r, w, k, v, a, b, ckpt, scratch, 16, dy, dsT, dr, dw, dk, dv, da, db,
                         ds0, stream);
}
