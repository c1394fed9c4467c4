// Direct-load kernel for sm_103a: the exact 2x uint8 downscale with every
// thread loading its own source bytes.
//
// For one frame per launch the path is bound by how fast HBM requests get in
// flight after the launch, not by bandwidth: a thread per output group, each
// with two 16- or 24-byte vector loads in flight at once (half a million
// threads for a 4K frame), reaches HBM sooner than a producer warp per CTA
// issuing bulk copies, and there is no stage to plan, no shared memory and
// no barrier.  Each thread forms one group of output pixels (8, 4 or 2
// pixels for 1, 3 or 4 channels) from the two source rows below it with the
// same exact arithmetic as the staged kernel (down2_group: (t0 + t1 + b0 + b1
// + 2) >> 2, CUDA interpolation page §2.2 and §6.2 at A = B = 1024), and
// writes it with one vector store.  Loads and stores bypass L1 and are
// evicted first from L2 (each byte is used once).
//
// Launched as a programmatic dependent launch: the grid may start while the
// previous kernel in the stream finishes, and waits (griddepcontrol.wait)
// before touching memory.
#include <cuda_runtime.h>

#include <cstdint>

#include "rz_device.h"
#include "rz_internal.h"

namespace rz {
namespace {

using namespace dev;

// Grid: x covers one image's output groups (kDirectThreads per CTA), y walks
// the images of a batch (strided past 65535 images).  Requirements, checked
// by the host: W = 2 OW, H = 2 OH; source base, pitch and batch stride
// multiples of the load width (16 bytes for 1 and 4 channels, 8 for 3);
// output base, pitch and batch stride multiples of the store width (8, 4).
template <int C>
__global__ void __launch_bounds__(kDirectThreads) k_down2_direct(const KArgs a, const __grid_constant__ CUtensorMap)
{
    constexpr int PX = down2_px(C);       // output pixels per group
    constexpr int SB = 2 * PX * C;        // source bytes per row and group: 16, 24, 16
    constexpr int OB = PX * C;            // output bytes per group: 8, 12, 8
    grid_launch_dependents();
    grid_dependency_wait();
    const int full = a.OW / PX;                // whole groups per row
    const int gpr = full + (a.OW % PX ? 1 : 0);
    const int idx = blockIdx.x * kDirectThreads + threadIdx.x;
    if (idx >= a.OH * gpr)
        return;
    const int dy = idx / gpr, j = idx - dy * gpr;
    for (int b = blockIdx.y; b < a.batch; b += gridDim.y) {
        const uint8_t *top = a.src + (long long)b * a.src_bstride + (long long)(2 * dy) * a.src_pitch;
        const uint8_t *bot = top + a.src_pitch;
        uint8_t *out = a.dst + (long long)b * a.dst_bstride + (long long)dy * a.dst_pitch;
        if (j < full) {
            uint32_t tw[SB / 4], bw[SB / 4], o[OB / 4];
            if constexpr (C == 3) {
                const uint2 *tp = reinterpret_cast<const uint2 *>(top + SB * j);
                const uint2 *bp = reinterpret_cast<const uint2 *>(bot + SB * j);
#pragma unroll
                for (int k = 0; k < 3; k++) {
                    const uint2 t = __ldcs(tp + k), u = __ldcs(bp + k);
                    tw[2 * k] = t.x; tw[2 * k + 1] = t.y;
                    bw[2 * k] = u.x; bw[2 * k + 1] = u.y;
                }
            } else {
                const uint4 t = __ldcs(reinterpret_cast<const uint4 *>(top + SB * j));
                const uint4 u = __ldcs(reinterpret_cast<const uint4 *>(bot + SB * j));
                tw[0] = t.x; tw[1] = t.y; tw[2] = t.z; tw[3] = t.w;
                bw[0] = u.x; bw[1] = u.y; bw[2] = u.z; bw[3] = u.w;
            }
            down2_group<C>(tw, bw, o);
            if constexpr (C == 3) {
                uint32_t *op = reinterpret_cast<uint32_t *>(out + OB * j);
                __stcs(op, o[0]);
                __stcs(op + 1, o[1]);
                __stcs(op + 2, o[2]);
            } else {
                __stcs(reinterpret_cast<uint2 *>(out + OB * j), make_uint2(o[0], o[1]));
            }
        } else {
            // the row's last pixels, fewer than a group: byte by byte
            for (int p = full * PX; p < a.OW; p++)
#pragma unroll
                for (int c = 0; c < C; c++) {
                    const int o = 2 * p * C + c;
                    const int s = top[o] + top[o + C] + bot[o] + bot[o + C] + 2;
                    out[p * C + c] = static_cast<uint8_t>(s >> 2);
                }
        }
    }
}

}  // namespace

const void *direct_down2_kernel_for(int C)
{
    using Fn = void (*)(const KArgs, const CUtensorMap);
    static const Fn k[3] = {k_down2_direct<1>, k_down2_direct<3>, k_down2_direct<4>};
    const int ci = (C == 1) ? 0 : (C == 3 ? 1 : (C == 4 ? 2 : -1));
    return ci < 0 ? nullptr : reinterpret_cast<const void *>(k[ci]);
}

}  // namespace rz
