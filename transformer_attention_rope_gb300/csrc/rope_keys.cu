// rope_keys.cu -- rotate keys into a pre-rotated KV cache (Part 1, §4.2-§4.4).
//
// Each pair (x_2i, x_2i+1) of the key at position pos0 + s is rotated by the
// table's (cos, sin)((pos0 + s) theta_i) in fp32 and stored as bf16; a thread
// handles one 16-byte chunk (4 pairs) of a row for up to eight heads.
#include "device_common.cuh"

namespace apex {
namespace {

// Each thread takes one 16-byte chunk position (s, c) and up to kHeads heads:
// the (cos, sin) values are read once and reused for every head (the table is
// otherwise re-read from L2 once per head).  Consecutive threads take
// consecutive chunks of a head, so the key loads and stores stay contiguous.
constexpr int kHeads = 8;
template <int LOG2C>
__global__ void __launch_bounds__(256) rope_keys_kernel(const RopeKeysParams p)
{
    constexpr int kChunks = 1 << LOG2C;
    constexpr int kHalf = 4 * kChunks;
    // launched as a programmatic dependent: the keys may be the previous
    // kernel's output, so nothing is read before that kernel is done
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int per_head = p.n_pos * kChunks;
    const int h_groups = (p.n_heads + kHeads - 1) / kHeads;
    for (int hg = blockIdx.y; hg < h_groups; hg += gridDim.y) {
        const int h0 = hg * kHeads;
        const int nh = min(kHeads, p.n_heads - h0);
        for (int idx = blockIdx.x * 256 + threadIdx.x; idx < per_head; idx += gridDim.x * 256) {
            const int c = idx & (kChunks - 1), s = idx >> LOG2C;
            const float4 *cs = reinterpret_cast<const float4 *>(p.rope.cs + (size_t)(p.pos0 + s) * kHalf + 4 * c);
            const float4 a = __ldg(cs), b = __ldg(cs + 1);
            uint4 v[kHeads];
#pragma unroll
            for (int j = 0; j < kHeads; ++j)
                if (j < nh) v[j] = *reinterpret_cast<const uint4 *>(p.in + (long long)(h0 + j) * p.in_stride + (size_t)idx * 8);
#pragma unroll
            for (int j = 0; j < kHeads; ++j)
                if (j < nh) {
                    uint4 o;
                    o.x = rope_pair_bf16(v[j].x, a.x, a.y);
                    o.y = rope_pair_bf16(v[j].y, a.z, a.w);
                    o.z = rope_pair_bf16(v[j].z, b.x, b.y);
                    o.w = rope_pair_bf16(v[j].w, b.z, b.w);
                    *reinterpret_cast<uint4 *>(p.out + (long long)(h0 + j) * p.out_stride + (size_t)idx * 8) = o;
                }
        }
    }
}

}  // namespace

cudaError_t launch_rope_keys(const RopeKeysParams &p, int sm_count, cudaStream_t stream)
{
    const int per_head = p.n_pos * (p.d_h / 8);
    const int h_groups = (p.n_heads + kHeads - 1) / kHeads;
    const int target = sm_count * 8;
    const int gy = h_groups < 65535 ? h_groups : 65535;
    int gx = (per_head + 255) / 256;
    const int gx_want = (target + gy - 1) / gy;
    if (gx > gx_want) gx = gx_want;
    // a programmatic dependent of the stream's previous work: the launch
    // overlaps that work's tail (the kernel waits for it before reading)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gx > 0 ? gx : 1, gy > 0 ? gy : 1);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.d_h == 128) return cudaLaunchKernelEx(&cfg, rope_keys_kernel<4>, p);
    if (p.d_h == 64) return cudaLaunchKernelEx(&cfg, rope_keys_kernel<3>, p);
    return cudaErrorInvalidValue;
}

}  // namespace apex
