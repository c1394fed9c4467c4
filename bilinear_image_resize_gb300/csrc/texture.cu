// Bilinear resize through the texture unit's hardware filtering, kept as a
// measured comparison with the exact kernels ("From Prototype to Performance:
// Optimizing OpenCV Resize on Volcanic GPUs", *Naive resize with linear
// sampling*: the sampler with unnormalised coordinates, texel centres at
// +0.5, sampled at (dst + 0.5) * in / out; CUDA interpolation page §4.1,
// texture memory with hardware interpolation).
//
// The texture unit forms the weights in low-precision fixed point (about 8
// fractional bits), so the result is not the exact 11-bit one: it may differ
// from the oracle by a unit or so, which the tests measure and bound.  The
// source is the caller's pitched uint8 image with 1 or 4 channels (there is
// no three-channel texture format), read as normalised floats and written
// back rounded to the nearest uint8.
#include <cuda_runtime.h>

#include <cstdint>
#include <new>

#include "rz_device.h"
#include "rz_internal.h"

struct rz_tex_s {
    cudaTextureObject_t tex = 0;
    int H = 0, W = 0, C = 0, device = 0;
};

namespace rz {
namespace {

// A thread per output pixel; the sampled point in texel units is
// (d + 0.5) * scale on each axis (the texture's own -0.5 puts it at the
// half-pixel position between texel centres).
template <int C>
__global__ void __launch_bounds__(256) k_tex_resize(cudaTextureObject_t tex, uint8_t *dst, long long dst_pitch,
                                                    int OH, int OW, float sx, float sy)
{
    dev::grid_launch_dependents();
    dev::grid_dependency_wait();
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= static_cast<long long>(OH) * OW)
        return;
    const int dy = static_cast<int>(idx / OW), dx = static_cast<int>(idx - static_cast<long long>(dy) * OW);
    const float fx = (static_cast<float>(dx) + 0.5f) * sx, fy = (static_cast<float>(dy) + 0.5f) * sy;
    uint8_t *op = dst + static_cast<long long>(dy) * dst_pitch + static_cast<long long>(dx) * C;
    if constexpr (C == 1) {
        const float v = tex2D<float>(tex, fx, fy);
        *op = static_cast<uint8_t>(__float2int_rn(v * 255.0f));
    } else {
        const float4 v = tex2D<float4>(tex, fx, fy);
        const uint32_t w = dev::pack4(__float2int_rn(v.x * 255.0f), __float2int_rn(v.y * 255.0f),
                                      __float2int_rn(v.z * 255.0f), __float2int_rn(v.w * 255.0f));
        if ((reinterpret_cast<uintptr_t>(op) & 3) == 0)
            *reinterpret_cast<uint32_t *>(op) = w;
        else
            for (int c = 0; c < 4; c++)
                op[c] = static_cast<uint8_t>(w >> (8 * c));
    }
}

}  // namespace
}  // namespace rz

extern "C" {

int resize_texture_create(rz_tex *out, const uint8_t *src, size_t src_pitch, int H, int W, int C)
{
    if (!out) return RZ_ERR_ARG;
    *out = nullptr;
    if (!src || H < 1 || W < 1 || H > RZ_MAX_DIM || W > RZ_MAX_DIM) return RZ_ERR_ARG;
    if (C != 1 && C != 4) return C < 1 ? RZ_ERR_ARG : RZ_ERR_UNSUPPORTED;
    if (src_pitch < static_cast<size_t>(W) * C) return RZ_ERR_ARG;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { rz::record_cuda_error(e); return RZ_ERR_CUDA; }
    int base_align = 0, pitch_align = 0;
    e = cudaDeviceGetAttribute(&base_align, cudaDevAttrTextureAlignment, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&pitch_align, cudaDevAttrTexturePitchAlignment, dev);
    if (e != cudaSuccess) { rz::record_cuda_error(e); return RZ_ERR_CUDA; }
    if ((reinterpret_cast<uintptr_t>(src) % static_cast<uintptr_t>(base_align)) != 0 ||
        src_pitch % static_cast<size_t>(pitch_align) != 0)
        return RZ_ERR_ARG;
    cudaResourceDesc rd = {};
    rd.resType = cudaResourceTypePitch2D;
    rd.res.pitch2D.devPtr = const_cast<uint8_t *>(src);
    rd.res.pitch2D.desc = C == 1 ? cudaCreateChannelDesc<unsigned char>() : cudaCreateChannelDesc<uchar4>();
    rd.res.pitch2D.width = static_cast<size_t>(W);
    rd.res.pitch2D.height = static_cast<size_t>(H);
    rd.res.pitch2D.pitchInBytes = src_pitch;
    cudaTextureDesc td = {};
    td.addressMode[0] = cudaAddressModeClamp;
    td.addressMode[1] = cudaAddressModeClamp;
    td.filterMode = cudaFilterModeLinear;
    td.readMode = cudaReadModeNormalizedFloat;
    td.normalizedCoords = 0;
    rz_tex_s *t = new (std::nothrow) rz_tex_s();
    if (!t) return RZ_ERR_NOMEM;
    e = cudaCreateTextureObject(&t->tex, &rd, &td, nullptr);
    if (e != cudaSuccess) {
        delete t;
        rz::record_cuda_error(e);
        return RZ_ERR_CUDA;
    }
    t->H = H; t->W = W; t->C = C; t->device = dev;
    *out = t;
    return RZ_OK;
}

int resize_texture_u8(rz_tex t, uint8_t *dst, size_t dst_pitch, int out_h, int out_w, void *stream)
{
    if (!t || out_h < 0 || out_w < 0 || out_h > RZ_MAX_DIM || out_w > RZ_MAX_DIM) return RZ_ERR_ARG;
    if (out_h == 0 || out_w == 0) return RZ_OK;
    if (!dst || dst_pitch < static_cast<size_t>(out_w) * t->C) return RZ_ERR_ARG;
    const float sx = static_cast<float>(static_cast<double>(t->W) / out_w);
    const float sy = static_cast<float>(static_cast<double>(t->H) / out_h);
    const long long n = static_cast<long long>(out_h) * out_w;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((n + 255) / 256), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const long long pitch = static_cast<long long>(dst_pitch);
    const cudaError_t e = t->C == 1
        ? cudaLaunchKernelEx(&cfg, rz::k_tex_resize<1>, t->tex, dst, pitch, out_h, out_w, sx, sy)
        : cudaLaunchKernelEx(&cfg, rz::k_tex_resize<4>, t->tex, dst, pitch, out_h, out_w, sx, sy);
    if (e != cudaSuccess) { rz::record_cuda_error(e); return RZ_ERR_CUDA; }
    return RZ_OK;
}

int resize_texture_destroy(rz_tex t)
{
    if (!t) return RZ_OK;
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != t->device) cudaSetDevice(t->device);
    // no queued kernel may still sample it
    cudaError_t e = cudaDeviceSynchronize();
    const cudaError_t e2 = cudaDestroyTextureObject(t->tex);
    if (e == cudaSuccess) e = e2;
    if (cur >= 0 && cur != t->device) cudaSetDevice(cur);
    delete t;
    if (e != cudaSuccess) { rz::record_cuda_error(e); return RZ_ERR_CUDA; }
    return RZ_OK;
}

}  // extern "C"
