// rope_keys.cu -- rotate keys into a pre-rotated KV cache (Part 1, §4.2-§4.4).
//
// One thread per 16-byte chunk (4 interleaved pairs) of a key row: threads with
// consecutive indices take consecutive chunks of a row, so loads and stores are
// contiguous.  Each pair (x_2i, x_2i+1) of the key at position pos0 + s is
// rotated by the table's (cos, sin)(pos * theta_i) in fp32 and stored as bf16.
#include "device_common.cuh"

namespace apex {
namespace {

__global__ void __launch_bounds__(256) rope_keys_kernel(const RopeKeysParams p)
{
    const int chunks = p.d_h / 8;
    const long long total = (long long)p.n_heads * p.n_pos * chunks;
    const int half = p.d_h / 2;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(idx % chunks);
        const long long rest = idx / chunks;
        const int s = (int)(rest % p.n_pos);
        const long long h = rest / p.n_pos;
        const uint4 v = *reinterpret_cast<const uint4 *>(p.in + h * p.in_stride + (long long)s * p.d_h + 8 * c);
        const float4 *cs = reinterpret_cast<const float4 *>(p.rope.cs + (size_t)(p.pos0 + s) * half + 4 * c);
        const float4 a = __ldg(cs), b = __ldg(cs + 1);
        uint4 r;
        r.x = rope_pair_bf16(v.x, a.x, a.y);
        r.y = rope_pair_bf16(v.y, a.z, a.w);
        r.z = rope_pair_bf16(v.z, b.x, b.y);
        r.w = rope_pair_bf16(v.w, b.z, b.w);
        *reinterpret_cast<uint4 *>(p.out + h * p.out_stride + (long long)s * p.d_h + 8 * c) = r;
    }
}

}  // namespace

cudaError_t launch_rope_keys(const RopeKeysParams &p, int sm_count, cudaStream_t stream)
{
    const long long total = (long long)p.n_heads * p.n_pos * (p.d_h / 8);
    const long long want = (total + 255) / 256;
    const int grid = (int)(want < (long long)sm_count * 8 ? want : (long long)sm_count * 8);
    rope_keys_kernel<<<grid > 0 ? grid : 1, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace apex
