// apex_attn_host.cu -- the C ABI of include/apex_attn.h: argument checks, the
// per-device RoPE cos/sin table, TMA descriptors and kernel launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "../../include/apex_attn.h"
#include "kernel_params.h"

namespace apex {

uint64_t wait_timeout_ns()
{
    static uint64_t v = [] {
        const char *e = getenv("APEX_ATTN_WAIT_TIMEOUT_MS");
        long ms = e ? atol(e) : 0;
        if (ms <= 0) ms = 2000;
        return (uint64_t)ms * 1000000ull;
    }();
    return v;
}

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSeq = 1 << 24;

// RoPE frequency parameters: base and the YaRN scaling (s <= 1: none).
struct RopeFreq {
    float base, yarn_s, beta_fast, beta_slow;
    bool operator==(const RopeFreq &o) const
    {
        return base == o.base && yarn_s == o.yarn_s && beta_fast == o.beta_fast && beta_slow == o.beta_slow;
    }
};

struct RopeTable {
    int d_h;
    RopeFreq f;
    float2 *dev;
    int cap;  // positions held
};

struct SplitPlan {
    int n_split, stages_per_split;
};

struct DeviceState {
    std::mutex mu;
    bool ready = false;
    int sm_count = 0;
    uint32_t *status = nullptr;  // per-device status word
    std::vector<RopeTable> tables;
    // last decode split plan: (units, stages, capacity) -> plan; the search
    // walks every split count, which for one sequence of 32K keys is ~500 steps
    int plan_key[3] = {-1, -1, -1};
    SplitPlan plan{1, 1};
};

DeviceState g_state[kMaxDevices];

// Prefill kernel choice for the plain block: the CTA-pair kernel for d_h = 128
// (measured 12 % faster than the single-CTA kernel on the B4 H_q32 H_kv8 S4096
// W1024 workload), the single-CTA kernel for d_h = 64 or when
// APEX_ATTN_PREFILL=single (read at each call).
bool use_pair_prefill(int d_h, int sm_count)
{
    const char *e = getenv("APEX_ATTN_PREFILL");
    if (e && strcmp(e, "single") == 0) return false;
    return d_h == 128 && sm_count >= 2;
}

apex_status init_device(DeviceState &st, int dev)
{
    if (st.ready) return APEX_OK;
    if (cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return APEX_ERR_CUDA;
    if (cudaMalloc(&st.status, sizeof(uint32_t)) != cudaSuccess) return APEX_ERR_NO_MEMORY;
    if (cudaMemset(st.status, 0, sizeof(uint32_t)) != cudaSuccess) return APEX_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return APEX_ERR_CUDA;
    st.ready = true;
    return APEX_OK;
}

// Part 1, §4.3: theta_i = base^(-2i/d_h); with YaRN (Part 1, §5.3-§5.4) the
// pair's wavelength 2 pi / theta_i decides: below beta_fast it is kept, above
// beta_slow * s it is divided by s, in between divided by t s + 1 - t with
// t = (wavelength / beta_slow - 1) / (s - 1) clamped to [0, 1].
double rope_frequency(int i, int d_h, const RopeFreq &f)
{
    const double theta = pow((double)f.base, -2.0 * (double)i / (double)d_h);
    if (!(f.yarn_s > 1.f)) return theta;
    const double s = f.yarn_s, lambda = 2.0 * 3.14159265358979323846 / theta;
    if (lambda < f.beta_fast) return theta;
    if (lambda > (double)f.beta_slow * s) return theta / s;
    double t = (lambda / f.beta_slow - 1.0) / (s - 1.0);
    t = t < 0.0 ? 0.0 : (t > 1.0 ? 1.0 : t);
    return theta / (t * s + (1.0 - t));
}

// Part 1, §5.5: the YaRN attention temperature multiplied into the scores.
double score_temperature(const RopeFreq &f) { return f.yarn_s > 1.f ? 0.1 * log((double)f.yarn_s) + 1.0 : 1.0; }

// Part 1, §4.7: the (cos, sin) cache of m * theta_i for every position m,
// computed in double precision and stored as fp32 pairs [cap][d_h/2].
apex_status get_table(DeviceState &st, int d_h, const RopeFreq &f, int need, RopeTableView *out)
{
    need = std::max(need, 128);
    for (auto &t : st.tables) {
        if (t.d_h == d_h && t.f == f && t.cap >= need) {
            *out = RopeTableView{t.dev, t.cap};
            return APEX_OK;
        }
    }
    int cap = 4096;
    while (cap < need) cap *= 2;
    const int half = d_h / 2;
    std::vector<float2> host((size_t)cap * half);
    for (int i = 0; i < half; ++i) {
        const double theta = rope_frequency(i, d_h, f);
        for (int m = 0; m < cap; ++m) {
            const double a = (double)m * theta;
            host[(size_t)m * half + i] = make_float2((float)cos(a), (float)sin(a));
        }
    }
    float2 *dev = nullptr;
    if (cudaMalloc(&dev, host.size() * sizeof(float2)) != cudaSuccess) {
        cudaGetLastError();
        return APEX_ERR_NO_MEMORY;
    }
    if (cudaMemcpy(dev, host.data(), host.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaFree(dev);
        return APEX_ERR_CUDA;
    }
    // replace a smaller table of the same parameters; cudaFree waits for the
    // device, so no kernel still reads the old one
    for (auto it = st.tables.begin(); it != st.tables.end(); ++it) {
        if (it->d_h == d_h && it->f == f) {
            cudaFree(it->dev);
            st.tables.erase(it);
            break;
        }
    }
    st.tables.push_back(RopeTable{d_h, f, dev, cap});
    *out = RopeTableView{dev, cap};
    return APEX_OK;
}

// Options -> frequency parameters, with the documented defaults; false when invalid.
bool freq_of(const apex_attn_options &o, RopeFreq *f)
{
    f->base = o.rope_base == 0.f ? 10000.f : o.rope_base;
    f->yarn_s = o.yarn_scale > 1.f ? o.yarn_scale : 1.f;
    f->beta_fast = o.yarn_beta_fast == 0.f ? 32.f : o.yarn_beta_fast;
    f->beta_slow = o.yarn_beta_slow == 0.f ? 1.f : o.yarn_beta_slow;
    if (!(f->base > 0.f) || !isfinite(f->base)) return false;
    if (!isfinite(o.yarn_scale) || !isfinite(f->yarn_s)) return false;
    if (f->yarn_s > 1.f && (!(f->beta_fast > 0.f) || !(f->beta_slow > 0.f) || !isfinite(f->beta_fast) ||
                            !isfinite(f->beta_slow)))
        return false;
    return true;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
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

// 3-D bf16 map over a dense [outer][rows][d_h] tensor, 128-byte swizzle, box
// {64 dims, box_rows, box_outer}; out-of-range elements read as zero.
bool make_map(CUtensorMap *m, const void *base, int d_h, int rows, int outer, int box_rows, int box_outer)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d_h, (cuuint64_t)rows, (cuuint64_t)outer};
    cuuint64_t strides[2] = {(cuuint64_t)d_h * 2, (cuuint64_t)rows * d_h * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_outer};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 4-D bf16 map over the output [units][G][S_q][128] of the CTA-pair prefill,
// box {64, min(P, 32), max(1, 32 / P), 1} with P = 128 / G (the 32 M-tile rows of
// one softmax warp, head-major), 128-byte swizzle.
bool make_out_map(CUtensorMap *m, void *base, int S_q, int G, int units)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const int P = 128 / G;
    cuuint64_t dims[4] = {128, (cuuint64_t)S_q, (cuuint64_t)G, (cuuint64_t)units};
    cuuint64_t strides[3] = {256, (cuuint64_t)S_q * 256, (cuuint64_t)G * S_q * 256};
    cuuint32_t box[4] = {64, (cuuint32_t)std::min(P, 32), (cuuint32_t)std::max(1, 32 / P), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_group(int G) { return G == 1 || G == 2 || G == 4 || G == 8 || G == 16; }

apex_status check_common(int B, int H_q, int H_kv, int S_k, int d_h, float base)
{
    if (B <= 0 || H_q <= 0 || H_kv <= 0 || S_k <= 0 || d_h <= 0) return APEX_ERR_INVALID_ARG;
    if (H_q % H_kv != 0) return APEX_ERR_INVALID_ARG;
    if (!(base > 0.f) || !isfinite(base)) return APEX_ERR_INVALID_ARG;
    if (S_k > kMaxSeq) return APEX_ERR_UNSUPPORTED;
    if (d_h != 64 && d_h != 128) return APEX_ERR_UNSUPPORTED;
    if (!supported_group(H_q / H_kv)) return APEX_ERR_UNSUPPORTED;
    if ((long long)B * H_q > (1ll << 30) || (long long)B * H_kv * (long long)S_k > (1ll << 40))
        return APEX_ERR_UNSUPPORTED;
    return APEX_OK;
}

DeviceState *current_state(int *dev_out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    *dev_out = dev;
    return &g_state[dev];
}

// --- decode split choice: the KV range of each (b, kv-head) unit is cut into
// n_split splits of whole 64-key stages; pick the count that minimises the
// modelled time rounds * (stages per split + 1) on a persistent grid.
int decode_split_cap(int units, int n_stages)
{
    long cap = std::max(1l, 32768l / std::max(1, units));
    cap = std::min<long>(cap, n_stages);
    cap = std::min<long>(cap, kDecodeMaxSplit);
    return (int)std::max(1l, cap);
}

SplitPlan plan_decode(int units, int n_stages, int capacity)
{
    const int cap = decode_split_cap(units, n_stages);
    SplitPlan best{1, n_stages};
    double best_cost = 1e300;
    for (int ns = 1; ns <= cap; ++ns) {
        const int sps = (n_stages + ns - 1) / ns;
        const int real = (n_stages + sps - 1) / sps;
        if (real != ns) continue;
        const long items = (long)units * ns;
        const long rounds = (items + capacity - 1) / capacity;
        const double cost = (double)rounds * (sps + 1);
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = SplitPlan{ns, sps};
        }
    }
    return best;
}

int max_stages_for(int S_k) { return (S_k + kDecodeKeysPerStage - 1) / kDecodeKeysPerStage + 1; }

// --- keys rotated once before the prefill.  Every work item of the prefill
// rotates the key tiles it visits (in shared memory); a key tile is visited
// by every item whose key range covers it, so it is rotated that many times
// (about 9 on B4 H_q32 S4096 W1024, 33 on S65536 W4096, 130 on a G = 16
// causal S8192).  Rotating the keys once into a workspace costs a read and a
// write of K.  Measured on GB300, plain 128-wide rows: about 1.7 ns of kernel
// time per (item, key tile) visit, against 10 ns per 128-key tile for the pass
// and about 1 us for its launch (the prefill, a programmatic dependent, sets up
// during the pass); decoupled-RoPE rows (128 + 64, only the 64-entry rope part
// turned): about 1.1 ns per visit against 15 ns per tile (1.5 times the bytes).
// The pass is used when it costs less than the visits it saves.
struct PrerotatePlan {
    bool use;
    int n_pos;  // keys rotated (whole 128-key tiles up to the last one any item reads)
};

// costs in units of 0.1 ns
struct PrerotateCost {
    int per_visit, per_tile;
};
constexpr PrerotateCost kCostPlain{17, 100};
constexpr PrerotateCost kCostDecoupled{11, 150};

PrerotatePlan plan_prerotate(int units, int S_q, int S_k, int q_pos0, int window, int P, int block_rows,
                             PrerotateCost cost)
{
    long long visits = 0;
    int kmax = 0;
    for (int r0 = 0; r0 < S_q; r0 += block_rows) {
        const int rows = std::min(block_rows, S_q - r0);
        const int m_first = q_pos0 + r0, m_last = q_pos0 + r0 + rows - 1;
        const int key_lo = (m_first < P || window <= 0) ? 0 : std::max(0, m_first - window + 1);
        const int key_hi = (m_first < P) ? std::max(m_last, P - 1) : m_last;
        visits += key_hi / 128 - key_lo / 128 + 1;
        kmax = std::max(kmax, key_hi);
    }
    const int n_pos = std::min(S_k, (kmax / 128 + 1) * 128);
    const long long tiles = (long long)units * ((n_pos + 127) / 128);
    visits *= units;
    return PrerotatePlan{visits * cost.per_visit >= tiles * cost.per_tile + 10000, n_pos};
}

}  // namespace
}  // namespace apex

using namespace apex;

extern "C" {

const char *apex_attn_status_string(apex_status s)
{
    switch (s) {
    case APEX_OK: return "ok";
    case APEX_ERR_INVALID_ARG: return "invalid argument";
    case APEX_ERR_UNSUPPORTED: return "unsupported configuration";
    case APEX_ERR_CUDA: return "CUDA error";
    case APEX_ERR_NO_MEMORY: return "out of device memory";
    case APEX_ERR_DEVICE_TIMEOUT: return "a kernel wait timed out";
    }
    return "unknown status";
}

apex_status apex_attn_rope_reserve(int max_pos, int d_h, float rope_base)
{
    if (max_pos <= 0 || max_pos > kMaxSeq) return APEX_ERR_INVALID_ARG;
    if (!(rope_base > 0.f) || !isfinite(rope_base)) return APEX_ERR_INVALID_ARG;
    if (d_h != 64 && d_h != 128) return APEX_ERR_UNSUPPORTED;
    int dev;
    DeviceState *st = current_state(&dev);
    if (!st) return APEX_ERR_CUDA;
    std::lock_guard<std::mutex> lk(st->mu);
    apex_status s = init_device(*st, dev);
    if (s != APEX_OK) return s;
    RopeTableView tv;
    return get_table(*st, d_h, RopeFreq{rope_base, 1.f, 32.f, 1.f}, max_pos, &tv);
}

apex_status apex_attn_device_status(void)
{
    int dev;
    DeviceState *st = current_state(&dev);
    if (!st) return APEX_ERR_CUDA;
    std::lock_guard<std::mutex> lk(st->mu);
    if (cudaDeviceSynchronize() != cudaSuccess) return APEX_ERR_CUDA;
    if (!st->ready) return APEX_OK;
    uint32_t v = 0;
    if (cudaMemcpy(&v, st->status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return APEX_ERR_CUDA;
    if (v == 0) return APEX_OK;
    if (cudaMemset(st->status, 0, sizeof(uint32_t)) != cudaSuccess) return APEX_ERR_CUDA;
    return APEX_ERR_DEVICE_TIMEOUT;
}

apex_status apex_attn_selftest_wait_timeout(int timeout_ms, apex_stream_t stream)
{
    if (timeout_ms < 1 || timeout_ms > 5000) return APEX_ERR_INVALID_ARG;
    int dev;
    DeviceState *st = current_state(&dev);
    if (!st) return APEX_ERR_CUDA;
    std::lock_guard<std::mutex> lk(st->mu);
    apex_status s = init_device(*st, dev);
    if (s != APEX_OK) return s;
    const WaitCtl wc{st->status, (uint64_t)timeout_ms * 1000000ull};
    if (launch_wait_selftest(wc, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return APEX_ERR_CUDA;
    return APEX_OK;
}

size_t apex_attn_decode_workspace_bytes(int B, int H_q, int H_kv, int S_k, int d_h)
{
    if (check_common(B, H_q, H_kv, S_k, d_h, 10000.f) != APEX_OK) return 0;
    const int units = B * H_kv;
    const int ns = decode_split_cap(units, max_stages_for(S_k));
    const size_t rows = (size_t)B * H_q * ns;
    size_t bytes = rows * (size_t)d_h * sizeof(float);
    bytes = (bytes + 15) & ~size_t(15);
    return bytes + rows * sizeof(float2);
}

// Decode of the plain block (d_qk = d_v = d_rope = d_h) or of decoupled-RoPE
// attention (d_qk = d_v + d_rope); argument checks of the callers done.
apex_status decode_launch(const void *q, const void *k_cache, const void *v_cache, void *out, int B, int H_q,
                          int H_kv, int S_k, int d_qk, int d_v, int d_rope, const apex_attn_options *opt,
                          const RopeFreq &f, void *workspace, size_t workspace_bytes, apex_stream_t stream)
{
    const int q_pos = opt->q_pos, window = opt->window, P = opt->prefix_len;
    if (q_pos < 0 || q_pos >= S_k) return APEX_ERR_INVALID_ARG;
    if (P < 0 || P > S_k) return APEX_ERR_INVALID_ARG;
    const size_t need = apex_attn_decode_workspace_bytes(B, H_q, H_kv, S_k, d_v);
    if (workspace_bytes < need) return APEX_ERR_INVALID_ARG;

    int dev;
    DeviceState *st = current_state(&dev);
    if (!st) return APEX_ERR_CUDA;
    std::lock_guard<std::mutex> lk(st->mu);
    apex_status s = init_device(*st, dev);
    if (s != APEX_OK) return s;
    RopeTableView tv;
    s = get_table(*st, d_rope, f, S_k, &tv);
    if (s != APEX_OK) return s;

    DecodeLaunch L;
    memset(&L, 0, sizeof L);
    const int units = B * H_kv;
    if (!make_map(&L.tm_k, k_cache, d_qk, S_k, units, kDecodeKeysPerStage, 1) ||
        !make_map(&L.tm_v, v_cache, d_v, S_k, units, kDecodeKeysPerStage, 1))
        return APEX_ERR_CUDA;
    DecodeParams &p = L.p;
    p.q = static_cast<const uint16_t *>(q);
    p.out = static_cast<uint16_t *>(out);
    const int ns_cap = decode_split_cap(units, max_stages_for(S_k));
    p.ws_o = static_cast<float *>(workspace);
    size_t o_bytes = (size_t)B * H_q * ns_cap * d_v * sizeof(float);
    o_bytes = (o_bytes + 15) & ~size_t(15);
    p.ws_ml = reinterpret_cast<float2 *>(static_cast<char *>(workspace) + o_bytes);
    p.rope = tv;
    p.wait = WaitCtl{st->status, wait_timeout_ns()};
    p.B = B;
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.G = H_q / H_kv;
    p.S_k = S_k;
    p.d_h = d_qk;
    p.d_v = d_v;
    p.d_rope = d_rope;
    p.q_pos = q_pos;
    // visible keys (Part 2, §10.2; a query inside the prefix sees the whole prefix, §11.1)
    if (q_pos < P) {
        p.k_lo = 0;
        p.k_hi = P - 1;
    } else {
        p.k_lo = (window > 0) ? std::max(0, q_pos - window + 1) : 0;
        p.k_hi = q_pos;
    }
    p.stage0 = p.k_lo / kDecodeKeysPerStage;
    p.n_stages = p.k_hi / kDecodeKeysPerStage - p.stage0 + 1;
    const int capacity = decode_ctas_per_sm(d_qk, d_v, p.G) * st->sm_count;
    if (st->plan_key[0] != units || st->plan_key[1] != p.n_stages || st->plan_key[2] != capacity) {
        st->plan = plan_decode(units, p.n_stages, capacity);
        st->plan_key[0] = units;
        st->plan_key[1] = p.n_stages;
        st->plan_key[2] = capacity;
    }
    const SplitPlan plan = st->plan;
    p.n_split = plan.n_split;
    p.stages_per_split = plan.stages_per_split;
    p.n_items = units * p.n_split;
    p.scale_log2 = (float)(1.4426950408889634 * score_temperature(f) / sqrt((double)d_qk));
    L.grid = std::min(p.n_items, capacity);
    if (launch_decode(L, opt->keys_prerotated != 0, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return APEX_ERR_CUDA;
    return APEX_OK;
}

apex_status apex_attn_decode_ex(const void *q, const void *k_cache, const void *v_cache, void *out, int B, int H_q,
                                int H_kv, int S_k, int d_h, const apex_attn_options *opt, void *workspace,
                                size_t workspace_bytes, apex_stream_t stream)
{
    if (!q || !k_cache || !v_cache || !out || !workspace || !opt) return APEX_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(workspace))
        return APEX_ERR_INVALID_ARG;
    RopeFreq f;
    if (!freq_of(*opt, &f)) return APEX_ERR_INVALID_ARG;
    apex_status s = check_common(B, H_q, H_kv, S_k, d_h, f.base);
    if (s != APEX_OK) return s;
    return decode_launch(q, k_cache, v_cache, out, B, H_q, H_kv, S_k, d_h, d_h, d_h, opt, f, workspace,
                         workspace_bytes, stream);
}

apex_status apex_attn_mla_decode(const void *q, const void *k_cache, const void *v_cache, void *out, int B, int H_q,
                                 int H_kv, int S_k, int d_h, int d_r, const apex_attn_options *opt, void *workspace,
                                 size_t workspace_bytes, apex_stream_t stream)
{
    if (!q || !k_cache || !v_cache || !out || !workspace || !opt) return APEX_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(workspace))
        return APEX_ERR_INVALID_ARG;
    if (d_r <= 0 || (d_r & 1)) return APEX_ERR_INVALID_ARG;
    RopeFreq f;
    if (!freq_of(*opt, &f)) return APEX_ERR_INVALID_ARG;
    apex_status s = check_common(B, H_q, H_kv, S_k, d_h, f.base);
    if (s != APEX_OK) return s;
    if (d_h != 128 || d_r != 64) return APEX_ERR_UNSUPPORTED;
    return decode_launch(q, k_cache, v_cache, out, B, H_q, H_kv, S_k, d_h + d_r, d_h, d_r, opt, f, workspace,
                         workspace_bytes, stream);
}

apex_status apex_attn_decode(const void *q, const void *k_cache, const void *v_cache, void *out, int B, int H_q,
                             int H_kv, int S_k, int d_h, int window, int q_pos, float rope_base, void *workspace,
                             size_t workspace_bytes, apex_stream_t stream)
{
    if (!(rope_base > 0.f)) return APEX_ERR_INVALID_ARG;
    apex_attn_options o;
    memset(&o, 0, sizeof o);
    o.window = window;
    o.q_pos = q_pos;
    o.rope_base = rope_base;
    return apex_attn_decode_ex(q, k_cache, v_cache, out, B, H_q, H_kv, S_k, d_h, &o, workspace, workspace_bytes,
                               stream);
}

// Prefill of the plain block (d_qk = d_v = d_rope = d_h) or of decoupled-RoPE
// attention (d_qk = d_v + d_rope): validation done by the callers.
apex_status prefill_launch(const void *q, const void *k, const void *v, void *out, int B, int H_q, int H_kv, int S_q,
                           int S_k, int d_qk, int d_v, int d_rope, const apex_attn_options *opt, const RopeFreq &f,
                           apex_stream_t stream, void *workspace = nullptr)
{
    const int q_pos0 = opt->q_pos, window = opt->window, P = opt->prefix_len;
    if (S_q <= 0 || q_pos0 < 0 || (long long)q_pos0 + S_q > (long long)S_k) return APEX_ERR_INVALID_ARG;
    if (P < 0 || P > S_k) return APEX_ERR_INVALID_ARG;

    int dev;
    DeviceState *st = current_state(&dev);
    if (!st) return APEX_ERR_CUDA;
    std::lock_guard<std::mutex> lk(st->mu);
    apex_status s = init_device(*st, dev);
    if (s != APEX_OK) return s;
    RopeTableView tv;
    s = get_table(*st, d_rope, f, S_k, &tv);
    if (s != APEX_OK) return s;

    const bool mla = d_qk != d_v;
    if (mla && st->sm_count < 2) return APEX_ERR_UNSUPPORTED;
    const int G = H_q / H_kv;
    const int rows_per_head = 128 / G;
    const bool pair = mla || use_pair_prefill(d_qk, st->sm_count);
    // keys rotated once into the workspace when that costs less than rotating
    // them in every work item that visits them
    PrerotatePlan pre{false, 0};
    if (workspace && !opt->keys_prerotated)
        pre = plan_prerotate(B * H_kv, S_q, S_k, q_pos0, window > 0 ? window : 0, P, (pair ? 4 : 2) * rows_per_head,
                             mla ? kCostDecoupled : kCostPlain);
    PrefillLaunch L;
    memset(&L, 0, sizeof L);
    if (!make_map(&L.tm_q, q, d_qk, S_q, B * H_q, rows_per_head, G) ||
        !make_map(&L.tm_k, pre.use ? workspace : k, d_qk, S_k, B * H_kv, pair ? 64 : 128, 1) ||
        !make_map(&L.tm_v, v, d_v, S_k, B * H_kv, 128, 1))
        return APEX_ERR_CUDA;
    if (pair && (d_v != 128 || !make_out_map(&L.tm_o, out, S_q, G, B * H_kv))) return APEX_ERR_CUDA;
    if (pre.use) {
        RopeKeysParams rp;
        rp.in = static_cast<const uint16_t *>(k);
        rp.out = static_cast<uint16_t *>(workspace);
        rp.in_stride = rp.out_stride = (long long)S_k * d_qk;
        rp.n_heads = B * H_kv;
        rp.n_pos = pre.n_pos;
        rp.d_row = d_qk;
        rp.d_rot = d_rope;
        rp.pos0 = 0;
        rp.rope = tv;
        if (launch_rope_keys(rp, st->sm_count, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
            return APEX_ERR_CUDA;
    }
    PrefillParams &p = L.p;
    p.out = static_cast<uint16_t *>(out);
    p.rope = tv;
    p.wait = WaitCtl{st->status, wait_timeout_ns()};
    p.B = B;
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.G = G;
    p.S_q = S_q;
    p.S_k = S_k;
    p.d_h = d_qk;
    p.d_rope = d_rope;
    p.window = window > 0 ? window : 0;
    p.q_pos0 = q_pos0;
    p.prefix_len = P;
    p.keys_prerotated = pre.use || opt->keys_prerotated != 0;
    p.rows_per_head = rows_per_head;
    const int block_rows = (pair ? 4 : 2) * rows_per_head;
    p.n_qblocks = (S_q + block_rows - 1) / block_rows;
    p.n_work = B * H_kv * p.n_qblocks;
    p.scale_log2 = (float)(1.4426950408889634 * score_temperature(f) / sqrt((double)d_qk));
    if (pair) {
        L.grid = 2 * std::min(p.n_work, st->sm_count / 2);
        if (launch_prefill_pair(L, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return APEX_ERR_CUDA;
    } else {
        L.grid = std::min(p.n_work, st->sm_count);
        if (launch_prefill(L, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return APEX_ERR_CUDA;
    }
    return APEX_OK;
}

apex_status apex_attn_fwd_ex(const void *q, const void *k, const void *v, void *out, int B, int H_q, int H_kv,
                             int S_q, int S_k, int d_h, const apex_attn_options *opt, apex_stream_t stream)
{
    if (!q || !k || !v || !out || !opt) return APEX_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return APEX_ERR_INVALID_ARG;
    RopeFreq f;
    if (!freq_of(*opt, &f)) return APEX_ERR_INVALID_ARG;
    apex_status s = check_common(B, H_q, H_kv, S_k, d_h, f.base);
    if (s != APEX_OK) return s;
    return prefill_launch(q, k, v, out, B, H_q, H_kv, S_q, S_k, d_h, d_h, d_h, opt, f, stream);
}

// Workspace of the key-rotation pass (0: the pass would not run); d_r = 0 for
// the plain block, else the rope part of decoupled-RoPE rows [d_h | d_r].
static size_t prefill_workspace_bytes(int B, int H_q, int H_kv, int S_q, int S_k, int d_h, int d_r,
                               const apex_attn_options *opt)
{
    if (!opt || opt->keys_prerotated) return 0;
    RopeFreq f;
    if (!freq_of(*opt, &f) || check_common(B, H_q, H_kv, S_k, d_h, f.base) != APEX_OK) return 0;
    if (d_r != 0 && (d_h != 128 || d_r != 64)) return 0;
    const int q_pos0 = opt->q_pos, P = opt->prefix_len;
    if (S_q <= 0 || q_pos0 < 0 || (long long)q_pos0 + S_q > (long long)S_k || P < 0 || P > S_k) return 0;
    // a work item covers 4 M tiles of 128 / G query rows on CTA pairs, 2 on one CTA
    const bool pair = d_r != 0 || use_pair_prefill(d_h, 2);
    const int block_rows = (pair ? 4 : 2) * (128 / (H_q / H_kv));
    const PrerotatePlan pr = plan_prerotate(B * H_kv, S_q, S_k, q_pos0, opt->window > 0 ? opt->window : 0, P,
                                            block_rows, d_r ? kCostDecoupled : kCostPlain);
    return pr.use ? (size_t)B * H_kv * (size_t)S_k * (d_h + d_r) * 2 : 0;
}

size_t apex_attn_fwd_workspace_bytes(int B, int H_q, int H_kv, int S_q, int S_k, int d_h,
                                     const apex_attn_options *opt)
{
    return prefill_workspace_bytes(B, H_q, H_kv, S_q, S_k, d_h, 0, opt);
}

size_t apex_attn_mla_fwd_workspace_bytes(int B, int H_q, int H_kv, int S_q, int S_k, int d_h, int d_r,
                                         const apex_attn_options *opt)
{
    if (d_r <= 0) return 0;
    return prefill_workspace_bytes(B, H_q, H_kv, S_q, S_k, d_h, d_r, opt);
}

apex_status apex_attn_fwd_ws(const void *q, const void *k, const void *v, void *out, int B, int H_q, int H_kv,
                             int S_q, int S_k, int d_h, const apex_attn_options *opt, void *workspace,
                             size_t workspace_bytes, apex_stream_t stream)
{
    if (!q || !k || !v || !out || !opt) return APEX_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return APEX_ERR_INVALID_ARG;
    RopeFreq f;
    if (!freq_of(*opt, &f)) return APEX_ERR_INVALID_ARG;
    apex_status s = check_common(B, H_q, H_kv, S_k, d_h, f.base);
    if (s != APEX_OK) return s;
    if (workspace &&
        (!aligned16(workspace) || workspace_bytes < apex_attn_fwd_workspace_bytes(B, H_q, H_kv, S_q, S_k, d_h, opt)))
        return APEX_ERR_INVALID_ARG;
    return prefill_launch(q, k, v, out, B, H_q, H_kv, S_q, S_k, d_h, d_h, d_h, opt, f, stream, workspace);
}

apex_status apex_attn_mla_fwd_ws(const void *q, const void *k, const void *v, void *out, int B, int H_q, int H_kv,
                                 int S_q, int S_k, int d_h, int d_r, const apex_attn_options *opt, void *workspace,
                                 size_t workspace_bytes, apex_stream_t stream)
{
    if (!q || !k || !v || !out || !opt) return APEX_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return APEX_ERR_INVALID_ARG;
    if (d_r <= 0 || (d_r & 1)) return APEX_ERR_INVALID_ARG;
    RopeFreq f;
    if (!freq_of(*opt, &f)) return APEX_ERR_INVALID_ARG;
    apex_status s = check_common(B, H_q, H_kv, S_k, d_h, f.base);
    if (s != APEX_OK) return s;
    if (d_h != 128 || d_r != 64) return APEX_ERR_UNSUPPORTED;
    if (workspace && (!aligned16(workspace) ||
                      workspace_bytes < apex_attn_mla_fwd_workspace_bytes(B, H_q, H_kv, S_q, S_k, d_h, d_r, opt)))
        return APEX_ERR_INVALID_ARG;
    return prefill_launch(q, k, v, out, B, H_q, H_kv, S_q, S_k, d_h + d_r, d_h, d_r, opt, f, stream, workspace);
}

apex_status apex_attn_mla_fwd(const void *q, const void *k, const void *v, void *out, int B, int H_q, int H_kv,
                              int S_q, int S_k, int d_h, int d_r, const apex_attn_options *opt, apex_stream_t stream)
{
    return apex_attn_mla_fwd_ws(q, k, v, out, B, H_q, H_kv, S_q, S_k, d_h, d_r, opt, nullptr, 0, stream);
}

apex_status apex_attn_fwd(const void *q, const void *k, const void *v, void *out, int B, int H_q, int H_kv,
                          int S_q, int S_k, int d_h, int window, int q_pos0, float rope_base, apex_stream_t stream)
{
    if (!(rope_base > 0.f)) return APEX_ERR_INVALID_ARG;
    apex_attn_options o;
    memset(&o, 0, sizeof o);
    o.window = window;
    o.q_pos = q_pos0;
    o.rope_base = rope_base;
    return apex_attn_fwd_ex(q, k, v, out, B, H_q, H_kv, S_q, S_k, d_h, &o, stream);
}

// Rows of d_row entries whose trailing d_rot entries are rotated (d_rot = d_row:
// the plain block; d_rot < d_row: the rope part of decoupled-RoPE rows).
static apex_status rope_keys_launch(const void *k_in, void *k_out, int n_heads, int n_pos, int d_row, int d_rot, int pos0,
                             long long in_head_stride, long long out_head_stride, const apex_attn_options *opt,
                             apex_stream_t stream)
{
    if (!k_in || !k_out || !opt) return APEX_ERR_INVALID_ARG;
    if (!aligned16(k_in) || !aligned16(k_out)) return APEX_ERR_INVALID_ARG;
    if (n_heads <= 0 || n_pos <= 0 || pos0 < 0) return APEX_ERR_INVALID_ARG;
    if (in_head_stride < (long long)n_pos * d_row || out_head_stride < (long long)n_pos * d_row ||
        (in_head_stride % 8) != 0 || (out_head_stride % 8) != 0)
        return APEX_ERR_INVALID_ARG;
    if ((long long)pos0 + n_pos > kMaxSeq) return APEX_ERR_UNSUPPORTED;
    RopeFreq f;
    if (!freq_of(*opt, &f)) return APEX_ERR_INVALID_ARG;
    int dev;
    DeviceState *st = current_state(&dev);
    if (!st) return APEX_ERR_CUDA;
    std::lock_guard<std::mutex> lk(st->mu);
    apex_status s = init_device(*st, dev);
    if (s != APEX_OK) return s;
    RopeTableView tv;
    s = get_table(*st, d_rot, f, pos0 + n_pos, &tv);
    if (s != APEX_OK) return s;
    RopeKeysParams p;
    p.in = static_cast<const uint16_t *>(k_in);
    p.out = static_cast<uint16_t *>(k_out);
    p.in_stride = in_head_stride;
    p.out_stride = out_head_stride;
    p.n_heads = n_heads;
    p.n_pos = n_pos;
    p.d_row = d_row;
    p.d_rot = d_rot;
    p.pos0 = pos0;
    p.rope = tv;
    if (launch_rope_keys(p, st->sm_count, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return APEX_ERR_CUDA;
    return APEX_OK;
}

apex_status apex_attn_rope_keys(const void *k_in, void *k_out, int n_heads, int n_pos, int d_h, int pos0,
                                long long in_head_stride, long long out_head_stride,
                                const apex_attn_options *opt, apex_stream_t stream)
{
    if (d_h != 64 && d_h != 128) return APEX_ERR_UNSUPPORTED;
    return rope_keys_launch(k_in, k_out, n_heads, n_pos, d_h, d_h, pos0, in_head_stride, out_head_stride, opt,
                            stream);
}

apex_status apex_attn_mla_rope_keys(const void *k_in, void *k_out, int n_heads, int n_pos, int d_h, int d_r,
                                    int pos0, long long in_head_stride, long long out_head_stride,
                                    const apex_attn_options *opt, apex_stream_t stream)
{
    if (d_r <= 0 || (d_r & 1)) return APEX_ERR_INVALID_ARG;
    if (d_h != 128 || d_r != 64) return APEX_ERR_UNSUPPORTED;
    return rope_keys_launch(k_in, k_out, n_heads, n_pos, d_h + d_r, d_r, pos0, in_head_stride, out_head_stride,
                            opt, stream);
}

}  // extern "C"
