// rope_keys.cu -- rotate keys into a pre-rotated KV cache (Part 1, §4.2-§4.4),
// or the rope part of decoupled-RoPE key rows [content | rope part] (Part 2,
// §9.3), whose content part is copied unchanged.
//
// Each pair (x_2i, x_2i+1) of the rotated part of the key at position pos0 + s
// is rotated by the table's (cos, sin)((pos0 + s) theta_i) in fp32 and stored
// as bf16, pairs numbered from the start of the rotated part; a thread handles
// one 16-byte chunk (4 pairs) of a row for up to eight heads.
#include "device_common.cuh"

namespace apex {
namespace {

// Each thread takes one 16-byte chunk position (s, c) and up to kHeads heads:
// the (cos, sin) values are read once and reused for every head (the table is
// otherwise re-read from L2 once per head).  Consecutive threads take
// consecutive chunks of a head, so the key loads and stores stay contiguous.
// CR: 16-byte chunks per row; the last CROT of them are rotated, the others copied.
constexpr int kHeads = 8;
template <int CR, int CROT>
__global__ void __launch_bounds__(256) rope_keys_kernel(const RopeKeysParams p)
{
    static_assert(CROT >= 1 && CROT <= CR, "rotated chunks");
    constexpr int kCopy = CR - CROT;
    constexpr int kHalf = 4 * CROT;  // pairs per table row
    // launched as a programmatic dependent: the keys may be the previous
    // kernel's output, so nothing is read before that kernel is done
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int per_head = p.n_pos * CR;
    const int h_groups = (p.n_heads + kHeads - 1) / kHeads;
    for (int hg = blockIdx.y; hg < h_groups; hg += gridDim.y) {
        const int h0 = hg * kHeads;
        const int nh = min(kHeads, p.n_heads - h0);
        for (int idx = blockIdx.x * 256 + threadIdx.x; idx < per_head; idx += gridDim.x * 256) {
            const int c = idx % CR, s = idx / CR;
            uint4 v[kHeads];
#pragma unroll
            for (int j = 0; j < kHeads; ++j)
                if (j < nh) v[j] = *reinterpret_cast<const uint4 *>(p.in + (long long)(h0 + j) * p.in_stride + (size_t)idx * 8);
            if (c < kCopy) {
#pragma unroll
                for (int j = 0; j < kHeads; ++j)
                    if (j < nh) *reinterpret_cast<uint4 *>(p.out + (long long)(h0 + j) * p.out_stride + (size_t)idx * 8) = v[j];
                continue;
            }
            const float4 *cs =
                reinterpret_cast<const float4 *>(p.rope.cs + (size_t)(p.pos0 + s) * kHalf + 4 * (c - kCopy));
            const float4 a = __ldg(cs), b = __ldg(cs + 1);
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
    const int per_head = p.n_pos * (p.d_row / 8);
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
    if (p.d_row == 128 && p.d_rot == 128) return cudaLaunchKernelEx(&cfg, rope_keys_kernel<16, 16>, p);
    if (p.d_row == 64 && p.d_rot == 64) return cudaLaunchKernelEx(&cfg, rope_keys_kernel<8, 8>, p);
    if (p.d_row == 192 && p.d_rot == 64) return cudaLaunchKernelEx(&cfg, rope_keys_kernel<24, 8>, p);
    return cudaErrorInvalidValue;
}

}  // namespace apex
