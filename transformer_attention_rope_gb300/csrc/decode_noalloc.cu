// decode_noalloc.cu -- apex_attn_decode_noalloc: the decode path with no device
// allocation at all, for callers that cannot allocate when they call us.
//
// Who needs it: code that runs where cudaMalloc is not an option -- an engine
// whose memory is fully carved up by its own pool at start-up (a direct
// cudaMalloc would fail, fragment the pool or stall on an implicit device
// synchronisation), a plugin ABI with a fixed signature that has no slot for a
// workspace pointer, or a latency-critical loop where an allocation's
// synchronisation is not acceptable.  For them, every byte this entry point
// touches besides the caller's q, caches and out lives in file-scope device
// arrays that exist from module load until process exit:
//   g_scratch  16 MiB   split-KV partial results (max, sum, unnormalised output)
//   g_rope     16 MiB   fp32 (cos, sin) table for positions < 32768, d_h <= 128
// The kernels are the same as apex_attn_decode's; only where the scratch and
// the table live differs.  Host code may only use the arrays' device addresses
// from cudaGetSymbolAddress: the array names themselves are host-side shadows.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "../../include/apex_attn.h"
#include "kernel_params.h"

namespace apex {
namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;
constexpr int kMaxPos = 32768;
constexpr int kMaxPairs = 64;  // d_h / 2 for d_h <= 128
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];
static __device__ __align__(256) float2 g_rope[kMaxPos * kMaxPairs];

struct NoAllocDevice {
    bool ready = false;
    unsigned char *scratch = nullptr;  // device address of g_scratch on this device
    float2 *rope = nullptr;            // device address of g_rope on this device
    int sm_count = 0;
    int table_d = 0;                   // (d_h, base) the table currently holds
    float table_base = 0.f;
};

std::mutex g_mu;
NoAllocDevice g_dev[kMaxDevices];

// (cos, sin)(m * theta_i), theta_i = base^(-2i/d_h), evaluated in double
// precision and stored as fp32 pairs [kMaxPos][d_h/2].
__global__ void rope_table_kernel(float2 *table, int d_h, double base)
{
    const int half = d_h / 2;
    const long n = (long)kMaxPos * half;
    for (long idx = blockIdx.x * (long)blockDim.x + threadIdx.x; idx < n; idx += (long)gridDim.x * blockDim.x) {
        const int m = (int)(idx / half), i = (int)(idx % half);
        const double a = (double)m * pow(base, -2.0 * (double)i / (double)d_h);
        double s, c;
        sincos(a, &s, &c);
        table[idx] = make_float2((float)c, (float)s);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [units][S_k][d_h] bf16, boxes of {64 dims, 64 keys, 1}, 128-byte swizzle, zero fill.
bool kv_map(CUtensorMap *m, const void *base, int d_h, int S_k, int units)
{
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d_h, (cuuint64_t)S_k, (cuuint64_t)units};
    cuuint64_t strides[2] = {(cuuint64_t)d_h * 2, (cuuint64_t)S_k * d_h * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kDecodeKeysPerStage, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t partial_bytes(int B, int H_q, int n_split, int d_h)
{
    const size_t rows = (size_t)B * H_q * n_split;
    size_t o = rows * (size_t)d_h * sizeof(float);
    o = (o + 15) & ~size_t(15);
    return o + rows * sizeof(float2);
}

}  // namespace
}  // namespace apex

using namespace apex;

extern "C" apex_status apex_attn_decode_noalloc(const void *q, const void *k_cache, const void *v_cache, void *out,
                                                int B, int H_q, int H_kv, int S_k, int d_h, int window, int q_pos,
                                                float rope_base, apex_stream_t stream)
{
    // ---- the same argument rules as apex_attn_decode ...
    if (!q || !k_cache || !v_cache || !out) return APEX_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return APEX_ERR_INVALID_ARG;
    if (B <= 0 || H_q <= 0 || H_kv <= 0 || S_k <= 0 || d_h <= 0 || H_q % H_kv != 0) return APEX_ERR_INVALID_ARG;
    if (!(rope_base > 0.f) || !isfinite(rope_base)) return APEX_ERR_INVALID_ARG;
    if (q_pos < 0 || q_pos >= S_k) return APEX_ERR_INVALID_ARG;
    const int G = H_q / H_kv;
    if (d_h != 64 && d_h != 128) return APEX_ERR_UNSUPPORTED;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return APEX_ERR_UNSUPPORTED;
    // ... plus the limits of the static arrays
    if (S_k > kMaxPos) return APEX_ERR_UNSUPPORTED;
    if ((long long)B * H_q > (1ll << 24) || partial_bytes(B, H_q, 1, d_h) > kScratchBytes) return APEX_ERR_UNSUPPORTED;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return APEX_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    NoAllocDevice &st = g_dev[dev];
    if (!st.ready) {
        // one-time set-up on this device: device addresses of the static arrays
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess) return APEX_ERR_CUDA;
        st.scratch = static_cast<unsigned char *>(p);
        if (cudaGetSymbolAddress(&p, g_rope) != cudaSuccess) return APEX_ERR_CUDA;
        st.rope = static_cast<float2 *>(p);
        if (cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return APEX_ERR_CUDA;
        st.ready = true;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (st.table_d != d_h || st.table_base != rope_base) {
        // (re)build the RoPE table for this (d_h, base), in stream order.  The
        // key is cleared first: if the launch or the wait fails, the array holds
        // a partly rewritten table that no later call may take for a valid one.
        st.table_d = 0;
        st.table_base = 0.f;
        rope_table_kernel<<<st.sm_count * 4, 256, 0, s>>>(st.rope, d_h, (double)rope_base);
        if (cudaGetLastError() != cudaSuccess) return APEX_ERR_CUDA;
        // finished before any later call, on any stream, reads it
        if (cudaStreamSynchronize(s) != cudaSuccess) return APEX_ERR_CUDA;
        st.table_d = d_h;
        st.table_base = rope_base;
    }

    DecodeLaunch L;
    memset(&L, 0, sizeof L);
    const int units = B * H_kv;
    if (!kv_map(&L.tm_k, k_cache, d_h, S_k, units) || !kv_map(&L.tm_v, v_cache, d_h, S_k, units))
        return APEX_ERR_CUDA;
    DecodeParams &p = L.p;
    p.q = static_cast<const uint16_t *>(q);
    p.out = static_cast<uint16_t *>(out);
    p.rope = RopeTableView{st.rope, kMaxPos};
    p.wait = WaitCtl{nullptr, wait_timeout_ns()};  // no status word: a time-out is not recorded
    p.B = B;
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.G = G;
    p.S_k = S_k;
    p.d_h = d_h;
    p.d_v = d_h;
    p.d_rope = d_h;
    p.q_pos = q_pos;
    p.k_lo = (window > 0) ? std::max(0, q_pos - window + 1) : 0;
    p.k_hi = q_pos;
    p.stage0 = p.k_lo / kDecodeKeysPerStage;
    p.n_stages = q_pos / kDecodeKeysPerStage - p.stage0 + 1;

    // splits: as many as the modelled time prefers, within what g_scratch holds
    int cap = (int)std::min<long>(std::max(1l, 32768l / units), (long)p.n_stages);
    while (cap > 1 && partial_bytes(B, H_q, cap, d_h) > kScratchBytes) --cap;
    const int capacity = decode_ctas_per_sm(d_h, d_h, G) * st.sm_count;
    int best_ns = 1, best_sps = p.n_stages;
    double best_cost = 1e300;
    for (int ns = 1; ns <= cap; ++ns) {
        const int sps = (p.n_stages + ns - 1) / ns;
        if ((p.n_stages + sps - 1) / sps != ns) continue;
        const long rounds = ((long)units * ns + capacity - 1) / capacity;
        const double cost = (double)rounds * (sps + 1);
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best_ns = ns;
            best_sps = sps;
        }
    }
    p.n_split = best_ns;
    p.stages_per_split = best_sps;
    p.n_items = units * p.n_split;
    size_t o_bytes = (size_t)B * H_q * p.n_split * d_h * sizeof(float);
    o_bytes = (o_bytes + 15) & ~size_t(15);
    p.ws_o = reinterpret_cast<float *>(st.scratch);
    p.ws_ml = reinterpret_cast<float2 *>(st.scratch + o_bytes);
    p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)d_h));
    L.grid = std::min(p.n_items, capacity);
    if (launch_decode(L, false, s) != cudaSuccess) return APEX_ERR_CUDA;
    return APEX_OK;
}
