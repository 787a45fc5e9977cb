// decode.cu -- single-query attention against a bf16 KV cache (sm_103a).
//
// The cache of one (batch, kv-head) unit is cut into 64-key stages and the
// stages into `n_split` contiguous splits.  A persistent grid of CTAs walks the
// (unit, split) items.  Per CTA:
//
//   warp 4 (producer): waits for a free ring slot, starts two TMA loads per
//       K / V box of the stage (128B-swizzled [64 keys][64 dims] boxes), then
//       rotates the G query vectors of the unit by R(q_pos - j0), j0 = first
//       key of the stage, and writes them to the slot as bf16.
//   warps 0-3 (consumers): each owns 16 of the 64 keys of every stage.  It
//       rotates its keys by R(j - j0) in registers straight after ldmatrix
//       (the offsets j - j0 are the same for every stage, so their cos/sin live
//       in registers), then runs S^T = K' Q'^T and O^T += V^T P^T on mma.sync
//       with fp32 accumulators and an online exp2 softmax.
//
// Rotating the query by -j0 and the key by its offset gives the same score as
// rotating both to their absolute positions, because a RoPE rotation by a
// followed by the inverse rotation by b is the rotation by a - b
// (<R(m) q, R(j) k> = <R(m - j0) q, R(j - j0) k>: Part 1, §4.5).
//
// At the end of an item the four warps merge their (max, sum, output) states
// in shared memory and write one partial per (b, h, split).  A second kernel
// merges the splits with a log-sum-exp reduction over warp shuffles.
//
// Query / key rows hold DQK entries, value / output rows DV; RoPE turns the
// trailing DR entries of the query and key rows (DQK = DV = DR for the plain
// block; DQK = DV + DR for decoupled RoPE, Part 2, §9.3, where the leading DV
// entries -- the content part -- are used as they are).
#include <math.h>

#include "device_common.cuh"

namespace apex {
namespace {

constexpr int kStages = 2;
constexpr int kKeys = kDecodeKeysPerStage;  // 64
constexpr int kBoxBytes = kKeys * 128;      // [64 keys][64 dims] bf16
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

template <int DQK, int DV, int NT>
struct DecodeCfg {
    static constexpr int kKBoxes = DQK / 64;
    static constexpr int kVBoxes = DV / 64;
    static constexpr int kKBytes = kKBoxes * kBoxBytes;
    static constexpr int kVBytes = kVBoxes * kBoxBytes;
    static constexpr int kQpRow = 2 * DQK + 16;  // padded row of the rotated queries
    static constexpr int kQpBytes = 8 * NT * kQpRow;
    static constexpr int kStageBytes = kKBytes + kVBytes + ((kQpBytes + 1023) / 1024) * 1024;
    static constexpr int kRedFloats = 8 * NT * (2 + DV);  // per warp: m, l, O[q][DV]
    static constexpr int kRedOff = kStages * kStageBytes;
    static constexpr int kBarOff = kRedOff + kConsumerWarps * kRedFloats * 4;
    static constexpr int kSmemBytes = kBarOff + 2 * kStages * 8 + 1024;  // + alignment slack
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap *m, uint32_t bar, int x, int y,
                                                 int z, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%3, %4, %5}], [%2], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(pol)
        : "memory");
}

// PREROT: the cached keys already hold RoPE(k_j, j); the query is rotated to
// its absolute position and the keys are used as they are.
template <int DQK, int DV, int DR, int NT, bool PREROT>
__global__ void __launch_bounds__(kThreads, 2)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const DecodeParams p)
{
    using C = DecodeCfg<DQK, DV, NT>;
    static_assert(DQK == DV + DR || (DQK == DV && DR == DQK), "row split");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + C::kBarOff;
    const uint32_t bar_empty = bar_full + 8 * kStages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 2);                 // producer: expect_tx + queries written
            mbar_init(bar_empty + 8 * s, kConsumerWarps);   // one arrival per consumer warp
        }
        fence_mbarrier_init();
    }
    // rows of the rotated-query area beyond G must read as zero
    for (int i = threadIdx.x; i < kStages * C::kQpBytes / 4; i += kThreads) {
        const int s = i / (C::kQpBytes / 4), w = i % (C::kQpBytes / 4);
        reinterpret_cast<uint32_t *>(smem + s * C::kStageBytes + C::kKBytes + C::kVBytes)[w] = 0u;
    }
    __syncthreads();
    // launched as a programmatic dependent: the set-up above overlaps the previous
    // kernel's tail; nothing in global memory is touched before that kernel is done
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
        }
        // the cache is streamed once: let its lines go first from L2
        uint64_t pol;
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
        constexpr int kPairs = DQK / 2;            // pairs of a query row
        constexpr int kCPairs = (DQK - DR) / 2;    // pairs of its content part (not rotated)
        constexpr int kRPairs = DR / 2;            // pairs of its rope part (table row length)
        constexpr int kPPL = (8 * NT * kPairs + 31) / 32;  // query pairs per lane
        const int n_pairs = p.G * kPairs;
        int it = 0;
        for (int item = blockIdx.x; item < p.n_items; item += gridDim.x) {
            const int split = item % p.n_split, unit = item / p.n_split;
            const int s_begin = p.stage0 + split * p.stages_per_split;
            const int s_end = min(p.stage0 + p.n_stages, s_begin + p.stages_per_split);
            // raw queries of the G heads of this unit (head h = unit*G + qi)
            float2 qv[kPPL];
#pragma unroll
            for (int k = 0; k < kPPL; ++k) {
                const int pi = lane + 32 * k;
                qv[k] = make_float2(0.f, 0.f);
                if (pi < n_pairs) {
                    const int qi = pi / kPairs, i = pi % kPairs;
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(
                        p.q + ((size_t)(unit * p.G + qi) * DQK + 2 * i));
                    qv[k] = make_float2(bf16lo_to_f32(w), bf16hi_to_f32(w));
                }
            }
            for (int st = s_begin; st < s_end; ++st, ++it) {
                const int slot = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                mbar_wait(bar_empty + 8 * slot, ph ^ 1, p.wait);
                const int j0 = st * kKeys;
                const uint32_t kdst = sbase + slot * C::kStageBytes;
                const uint32_t vdst = kdst + C::kKBytes;
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar_full + 8 * slot, C::kKBytes + C::kVBytes);
#pragma unroll
                    for (int bx = 0; bx < C::kKBoxes; ++bx)
                        tma_load_3d_hint(kdst + bx * kBoxBytes, &tm_k, bar_full + 8 * slot, 64 * bx, j0, unit, pol);
#pragma unroll
                    for (int bx = 0; bx < C::kVBoxes; ++bx)
                        tma_load_3d_hint(vdst + bx * kBoxBytes, &tm_v, bar_full + 8 * slot, 64 * bx, j0, unit, pol);
                }
                // Q' = R(q_pos - j0) q (Part 1, §4.2 rotation of each interleaved pair);
                // a query inside a prefix can see keys after it: R(-a) = (cos a, -sin a).
                // With pre-rotated keys, Q' = R(q_pos) q.
                const int delta = PREROT ? p.q_pos : p.q_pos - j0;
                const float2 *cs = p.rope.cs + (size_t)(delta < 0 ? -delta : delta) * kRPairs;
                const float sgn = delta < 0 ? -1.f : 1.f;
                uint8_t *qp = smem + slot * C::kStageBytes + C::kKBytes + C::kVBytes;
#pragma unroll
                for (int k = 0; k < kPPL; ++k) {
                    const int pi = lane + 32 * k;
                    if (pi < n_pairs) {
                        const int qi = pi / kPairs, i = pi % kPairs;
                        uint32_t word;
                        if (kCPairs > 0 && i < kCPairs) {
                            word = pack_bf16x2(qv[k].x, qv[k].y);  // content: exact bf16 copy
                        } else {
                            const float2 c0 = __ldg(cs + (i - kCPairs));
                            const float2 c = make_float2(c0.x, sgn * c0.y);
                            const float y0 = fmaf(qv[k].x, c.x, -qv[k].y * c.y);
                            const float y1 = fmaf(qv[k].x, c.y, qv[k].y * c.x);
                            word = pack_bf16x2(y0, y1);
                        }
                        *reinterpret_cast<uint32_t *>(qp + qi * C::kQpRow + 4 * i) = word;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_full + 8 * slot);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, t = lane & 3;
    constexpr int kRPairs = DR / 2;              // table row length
    constexpr int kRopeStep0 = (DQK - DR) / 16;  // first k-step of the rope part
    // cos/sin of the key offsets this thread rotates: rows r0 = 16w+g, r1 = r0+8;
    // in rope k-step sr the rope pairs 8sr+t (bits 0..7 of the step) and 8sr+4+t.
    float2 csk[2][DR / 8];
    {
        const int r0 = 16 * warp + g;
#pragma unroll
        for (int sr = 0; sr < DR / 16; ++sr)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int pair = 8 * sr + 4 * h + t;
                csk[0][2 * sr + h] = __ldg(p.rope.cs + (size_t)r0 * kRPairs + pair);
                csk[1][2 * sr + h] = __ldg(p.rope.cs + (size_t)(r0 + 8) * kRPairs + pair);
            }
    }
    float *red_all = reinterpret_cast<float *>(smem + C::kRedOff);
    float *red = red_all + warp * C::kRedFloats;

    int it = 0;
    for (int item = blockIdx.x; item < p.n_items; item += gridDim.x) {
        const int split = item % p.n_split, unit = item / p.n_split;
        const int s_begin = p.stage0 + split * p.stages_per_split;
        const int s_end = min(p.stage0 + p.n_stages, s_begin + p.stages_per_split);

        float m_run[NT][2], l_run[NT][2];
        float acc_o[DV / 16][NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                m_run[nt][c] = -INFINITY;
                l_run[nt][c] = 0.f;
            }
#pragma unroll
        for (int mt = 0; mt < DV / 16; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc_o[mt][nt][e] = 0.f;

        for (int st = s_begin; st < s_end; ++st, ++it) {
            const int slot = it % kStages;
            mbar_wait(bar_full + 8 * slot, (it / kStages) & 1, p.wait);
            const int j0 = st * kKeys;
            const uint32_t kb = sbase + slot * C::kStageBytes;
            const uint32_t vb = kb + C::kKBytes;
            const uint32_t qp = vb + C::kVBytes;

            // S^T[16 keys x 8NT queries] = K'[16 x DQK] . Q'^T[DQK x 8NT]
            float acc_s[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc_s[nt][e] = 0.f;
#pragma unroll
            for (int s2 = 0; s2 < DQK / 32; ++s2) {
                uint32_t bq[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    ldmatrix_x4(bq[nt], qp + (8 * nt + (lane & 7)) * C::kQpRow + (4 * s2 + (lane >> 3)) * 16);
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int s = 2 * s2 + h2;
                    const uint32_t row = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const uint32_t chunk = 2 * s + (lane >> 4);
                    uint32_t a[4];
                    ldmatrix_x4(a, kb + (chunk >> 3) * kBoxBytes + swz128(row, chunk & 7));
                    if (!PREROT && s >= kRopeStep0) {
                        const int sr = s - kRopeStep0;
                        a[0] = rope_pair_bf16(a[0], csk[0][2 * sr].x, csk[0][2 * sr].y);
                        a[1] = rope_pair_bf16(a[1], csk[1][2 * sr].x, csk[1][2 * sr].y);
                        a[2] = rope_pair_bf16(a[2], csk[0][2 * sr + 1].x, csk[0][2 * sr + 1].y);
                        a[3] = rope_pair_bf16(a[3], csk[1][2 * sr + 1].x, csk[1][2 * sr + 1].y);
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc_s[nt], a, bq[nt][2 * h2], bq[nt][2 * h2 + 1]);
                }
            }

            // online softmax over this warp's 16 keys (log2 units)
            const bool edge = (j0 < p.k_lo) || (j0 + kKeys - 1 > p.k_hi);
            const int key0 = j0 + 16 * warp + g, key1 = key0 + 8;
            const bool ok0 = !edge || (key0 >= p.k_lo && key0 <= p.k_hi);
            const bool ok1 = !edge || (key1 >= p.k_lo && key1 <= p.k_hi);
            uint32_t bp[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float pv[4];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const float s0 = ok0 ? acc_s[nt][c] * p.scale_log2 : -INFINITY;
                    const float s1 = ok1 ? acc_s[nt][c + 2] * p.scale_log2 : -INFINITY;
                    float mx = fmaxf(s0, s1);
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    const float m_new = fmaxf(m_run[nt][c], mx);
                    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                    const float alpha = fast_exp2(m_run[nt][c] - m_use);
                    pv[c] = fast_exp2(s0 - m_use);
                    pv[c + 2] = fast_exp2(s1 - m_use);
                    l_run[nt][c] = l_run[nt][c] * alpha + pv[c] + pv[c + 2];
                    m_run[nt][c] = m_new;
#pragma unroll
                    for (int mt = 0; mt < DV / 16; ++mt) {
                        acc_o[mt][nt][c] *= alpha;
                        acc_o[mt][nt][c + 2] *= alpha;
                    }
                }
                // P^T fragments (keys x queries) from the S^T accumulator layout
                bp[nt][0] = movmatrix_trans(pack_bf16x2(pv[0], pv[1]));
                bp[nt][1] = movmatrix_trans(pack_bf16x2(pv[2], pv[3]));
            }

            // O^T[DV x 8NT] += V^T[DV x 16 keys] . P^T[16 keys x 8NT]
#pragma unroll
            for (int mt = 0; mt < DV / 16; ++mt) {
                const uint32_t row = 16 * warp + (lane & 7) + (lane >> 4) * 8;
                const uint32_t chunk = 2 * mt + ((lane >> 3) & 1);
                uint32_t a[4];
                ldmatrix_x4_trans(a, vb + (chunk >> 3) * kBoxBytes + swz128(row, chunk & 7));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc_o[mt][nt], a, bp[nt][0], bp[nt][1]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
        }

        // ---- merge the four warps' states and write this split's partial
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float l = l_run[nt][c];
                l += __shfl_xor_sync(0xffffffffu, l, 4);
                l += __shfl_xor_sync(0xffffffffu, l, 8);
                l += __shfl_xor_sync(0xffffffffu, l, 16);
                const int qc = 8 * nt + 2 * t + c;
                if (g == 0) {
                    red[qc] = m_run[nt][c];
                    red[8 * NT + qc] = l;
                }
#pragma unroll
                for (int mt = 0; mt < DV / 16; ++mt) {
                    red[16 * NT + qc * DV + 16 * mt + g] = acc_o[mt][nt][c];
                    red[16 * NT + qc * DV + 16 * mt + g + 8] = acc_o[mt][nt][c + 2];
                }
            }
        named_bar_sync(1, kConsumerWarps * 32);
        for (int idx = threadIdx.x; idx < p.G * DV; idx += kConsumerWarps * 32) {
            const int qc = idx / DV, e = idx % DV;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, red_all[w * C::kRedFloats + qc]);
            if (M == -INFINITY) M = 0.f;
            float L = 0.f, O = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float *rw = red_all + w * C::kRedFloats;
                const float mw = rw[qc];
                const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
                L += f * rw[8 * NT + qc];
                O += f * rw[16 * NT + qc * DV + e];
            }
            const size_t slot_idx = (size_t)(unit * p.G + qc) * p.n_split + split;
            p.ws_o[slot_idx * DV + e] = O;
            if (e == 0) p.ws_ml[slot_idx] = make_float2(M, L);
        }
        named_bar_sync(1, kConsumerWarps * 32);
    }
}

// One warp per (b, h): log-sum-exp merge of the n_split partials.
template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeParams p)
{
    // launched as a programmatic dependent of the split kernel: every partial is
    // written and visible once this returns
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * 4 + warp;
    if (row >= p.B * p.H_q) return;
    const float2 *ml = p.ws_ml + (size_t)row * p.n_split;
    float M = -INFINITY;
    for (int s = lane; s < p.n_split; s += 32) M = fmaxf(M, ml[s].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (M == -INFINITY) M = 0.f;
    float L = 0.f;
    for (int s = lane; s < p.n_split; s += 32) {
        const float2 v = ml[s];
        L += (v.x == -INFINITY) ? 0.f : exp2f(v.x - M) * v.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);

    constexpr int E = D / 32;  // output dims per lane
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    const float *o = p.ws_o + (size_t)row * p.n_split * D + lane * E;
    for (int s = 0; s < p.n_split; ++s) {
        const float2 v = ml[s];
        const float w = (v.x == -INFINITY) ? 0.f : exp2f(v.x - M);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += w * o[(size_t)s * D + e];
    }
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    uint32_t packed[E / 2];
#pragma unroll
    for (int e = 0; e < E / 2; ++e) packed[e] = pack_bf16x2(acc[2 * e] * inv, acc[2 * e + 1] * inv);
    uint32_t *dst = reinterpret_cast<uint32_t *>(p.out + (size_t)row * D + lane * E);
#pragma unroll
    for (int e = 0; e < E / 2; ++e) dst[e] = packed[e];
}

template <int DQK, int DV, int DR, int NT, bool PREROT>
cudaError_t launch_t(const DecodeLaunch &L, cudaStream_t stream)
{
    using C = DecodeCfg<DQK, DV, NT>;
    cudaError_t err = cudaFuncSetAttribute(decode_split_kernel<DQK, DV, DR, NT, PREROT>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (err != cudaSuccess) return err;
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(L.grid);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = C::kSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        err = cudaLaunchKernelEx(&cfg, decode_split_kernel<DQK, DV, DR, NT, PREROT>, L.tm_k, L.tm_v, L.p);
        if (err != cudaSuccess) return err;
    }
    const int rows = L.p.B * L.p.H_q;
    // programmatic dependent launch: the combine grid's launch is prepared while
    // the split grid runs, and its blocks wait (griddepcontrol.wait) for that
    // grid's completion.  The split kernel does not signal early: a trigger at its
    // start measured 1-2 % slower at B = 16 and 64 (the waiting blocks took
    // resident slots); without one, B = 1 runs 6.5 % faster, B = 4 2.6 %.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((rows + 3) / 4);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel<DV>, L.p);
}

template <bool PREROT>
cudaError_t dispatch(const DecodeLaunch &L, cudaStream_t stream)
{
    const bool wide = L.p.G > 8;
    const int dqk = L.p.d_h, dv = L.p.d_v, dr = L.p.d_rope;
    if (dqk == 128 && dv == 128 && dr == 128)
        return wide ? launch_t<128, 128, 128, 2, PREROT>(L, stream) : launch_t<128, 128, 128, 1, PREROT>(L, stream);
    if (dqk == 64 && dv == 64 && dr == 64)
        return wide ? launch_t<64, 64, 64, 2, PREROT>(L, stream) : launch_t<64, 64, 64, 1, PREROT>(L, stream);
    if (dqk == 192 && dv == 128 && dr == 64)
        return wide ? launch_t<192, 128, 64, 2, PREROT>(L, stream) : launch_t<192, 128, 64, 1, PREROT>(L, stream);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(const DecodeLaunch &L, bool keys_prerotated, cudaStream_t stream)
{
    return keys_prerotated ? dispatch<true>(L, stream) : dispatch<false>(L, stream);
}

// Resident split-kernel CTAs per SM (the shared-memory footprint decides).
int decode_ctas_per_sm(int d_qk, int d_v, int G)
{
    const bool wide = G > 8;
    int bytes = 0;
    if (d_qk == 192 && d_v == 128)
        bytes = wide ? DecodeCfg<192, 128, 2>::kSmemBytes : DecodeCfg<192, 128, 1>::kSmemBytes;
    else if (d_qk == 128)
        bytes = wide ? DecodeCfg<128, 128, 2>::kSmemBytes : DecodeCfg<128, 128, 1>::kSmemBytes;
    else
        bytes = wide ? DecodeCfg<64, 64, 2>::kSmemBytes : DecodeCfg<64, 64, 1>::kSmemBytes;
    // 228 KB of shared memory per SM, 1 KB of it reserved per resident CTA
    const int n = (228 * 1024) / (bytes + 1024);
    return n < 1 ? 1 : (n > 2 ? 2 : n);
}

}  // namespace apex
