// prefill.cu -- RoPE + GQA + causal/sliding-window attention on tcgen05 (sm_103a).
//
// One CTA per work item (b, kv-head g, block of query positions).  The block
// holds two 128-row M tiles Q0, Q1.  Each M tile packs the G query heads that
// share KV head g (Part 2, §8.2): rows are head-major, G heads x P = 128/G
// consecutive positions, so one K/V tile feeds all G heads at once.
//
// Warp roles (14 warps):
//   0-3   softmax + epilogue of Q0 (thread i owns row i / TMEM lane i)
//   4-7   softmax + epilogue of Q1
//   8-11  RoPE: rotate Q0/Q1 once and every K tile in shared memory, in place,
//         on the 128B-swizzled TMA layout (Part 1, §4.2-§4.4)
//   12    TMA producer (Q once, then the K and V rings)
//   13    MMA issuer: S_t = Q_t K^T and O_t += P_t V on tcgen05, accumulators
//         in TMEM (S0, S1, O0, O1 = 512 columns), P_t written over S_t as bf16
//
// Only key tiles that hold at least one visible key of the block are visited
// (Part 2, §10.2-§10.3: the window makes the work O(S W)); per-element masking
// is applied only where a tile is not entirely visible to a row.  The softmax
// is the online form of Part 2, §6.2 in log2 units: a running max that is
// raised (and O, l rescaled) only when the new tile max exceeds it by more
// than 8, which leaves the final O / l unchanged.
#include <math.h>

#include "device_common.cuh"
#include "tcgen05.cuh"

namespace apex {
namespace {

constexpr int kThreads = 14 * 32;
constexpr int kWarpRope = 8;
constexpr int kWarpTma = 12;
constexpr int kWarpMma = 13;
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kBoxBytes = 128 * 128;  // [128 rows][64 bf16]

template <int D>
struct Cfg {
    static constexpr int kBoxes = D / 64;
    static constexpr int kTile = kBoxes * kBoxBytes;  // 128 x D bf16
    static constexpr int kQOff = 0;
    static constexpr int kKOff = 2 * kTile;
    static constexpr int kVOff = kKOff + kKStages * kTile;
    static constexpr int kBarOff = kVOff + kVStages * kTile;
    // barrier slots
    static constexpr int kBarQFull = 0;                       // [2]
    static constexpr int kBarQReady = 2;                      // [1]
    static constexpr int kBarKFull = 3;                       // [kKStages]
    static constexpr int kBarKReady = kBarKFull + kKStages;   // [kKStages]
    static constexpr int kBarKEmpty = kBarKReady + kKStages;  // [kKStages]
    static constexpr int kBarVFull = kBarKEmpty + kKStages;   // [kVStages]
    static constexpr int kBarVEmpty = kBarVFull + kVStages;   // [kVStages]
    static constexpr int kBarSFull = kBarVEmpty + kVStages;   // [2]
    static constexpr int kBarPReady = kBarSFull + 2;          // [2]
    static constexpr int kBarODone = kBarPReady + 2;          // [2]
    static constexpr int kNumBars = kBarODone + 2;
    static constexpr int kTmemSlot = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kTmemSlot + 16 + 1024;
    // TMEM columns: S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D)
    __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
    __device__ static constexpr uint32_t col_o(int t) { return 256u + (uint32_t)D * t; }
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Rotate rows [0, 128) of a 128 x D tile stored as D/64 swizzled boxes.
// Thread rt (0..127) takes 16-byte chunk (rt & 7) of rows (rt >> 3) + 16 k.
// pos_of(row) returns the position of a row, or -1 to leave the row as is.
template <int D, typename PosFn>
__device__ __forceinline__ void rope_tile(uint8_t *tile, int rt, const float2 *cs_table, PosFn pos_of)
{
    const int c = rt & 7;
#pragma unroll 2
    for (int k = 0; k < 8; ++k) {
        const int row = (rt >> 3) + 16 * k;
        const int pos = pos_of(row);
        if (pos < 0) continue;
        const float2 *cs_row = cs_table + (size_t)pos * (D / 2);
#pragma unroll
        for (int bx = 0; bx < D / 64; ++bx) {
            uint4 *ptr = reinterpret_cast<uint4 *>(tile + bx * kBoxBytes + swz128(row, c));
            uint4 v = *ptr;
            const float4 *cs4 = reinterpret_cast<const float4 *>(cs_row + bx * 32 + 4 * c);
            const float4 a = __ldg(cs4), b = __ldg(cs4 + 1);
            v.x = rope_pair_bf16(v.x, a.x, a.y);
            v.y = rope_pair_bf16(v.y, a.z, a.w);
            v.z = rope_pair_bf16(v.z, b.x, b.y);
            v.w = rope_pair_bf16(v.w, b.z, b.w);
            *ptr = v;
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const PrefillParams p)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) -> uint32_t { return sb + C::kBarOff + 8 * i; };

    // ---- work item, heaviest (latest positions) first
    const int units = p.B * p.H_kv;
    const int qblock = p.n_qblocks - 1 - (int)blockIdx.x / units;
    const int unit = (int)blockIdx.x % units;
    const int b = unit / p.H_kv, hk = unit % p.H_kv;
    const int P = p.rows_per_head;
    const int r0 = qblock * 2 * P;
    const int rows_in_block = min(2 * P, p.S_q - r0);
    const int m_first = p.q_pos0 + r0;
    const int m_last = p.q_pos0 + r0 + rows_in_block - 1;
    const int j_lo = (p.window > 0) ? max(0, m_first - p.window + 1) / 128 : 0;
    const int n_kt = m_last / 128 - j_lo + 1;
    const int zq = b * p.H_q + hk * p.G;

    if (threadIdx.x == 0) {
        mbar_init(bar(C::kBarQFull + 0), 1);
        mbar_init(bar(C::kBarQFull + 1), 1);
        mbar_init(bar(C::kBarQReady), 4);
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(bar(C::kBarKFull + s), 1);
            mbar_init(bar(C::kBarKReady + s), 4);
            mbar_init(bar(C::kBarKEmpty + s), 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(bar(C::kBarVFull + s), 1);
            mbar_init(bar(C::kBarVEmpty + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(C::kBarSFull + t), 1);
            mbar_init(bar(C::kBarPReady + t), 4);
            mbar_init(bar(C::kBarODone + t), 1);
        }
        fence_mbarrier_init();
    }
    if (warp == kWarpMma) tmem_alloc(sb + C::kTmemSlot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + C::kTmemSlot);

    if (warp == kWarpTma) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_o);
            for (int t = 0; t < 2; ++t) {
                mbar_arrive_expect_tx(bar(C::kBarQFull + t), C::kTile);
#pragma unroll
                for (int bx = 0; bx < C::kBoxes; ++bx)
                    tma_load_3d(sb + C::kQOff + t * C::kTile + bx * kBoxBytes, &tm_q, bar(C::kBarQFull + t),
                                64 * bx, r0 + t * P, zq);
            }
            for (int j = 0; j < n_kt; ++j) {
                const int key0 = 128 * (j_lo + j);
                const int ks = j % kKStages, vs = j % kVStages;
                mbar_wait(bar(C::kBarKEmpty + ks), ((j / kKStages) & 1) ^ 1, p.wait);
                mbar_arrive_expect_tx(bar(C::kBarKFull + ks), C::kTile);
#pragma unroll
                for (int bx = 0; bx < C::kBoxes; ++bx)
                    tma_load_3d(sb + C::kKOff + ks * C::kTile + bx * kBoxBytes, &tm_k, bar(C::kBarKFull + ks),
                                64 * bx, key0, unit);
                mbar_wait(bar(C::kBarVEmpty + vs), ((j / kVStages) & 1) ^ 1, p.wait);
                mbar_arrive_expect_tx(bar(C::kBarVFull + vs), C::kTile);
#pragma unroll
                for (int bx = 0; bx < C::kBoxes; ++bx)
                    tma_load_3d(sb + C::kVOff + vs * C::kTile + bx * kBoxBytes, &tm_v, bar(C::kBarVFull + vs),
                                64 * bx, key0, unit);
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
            auto issue_qk = [&](int t, int ks) {
                const uint32_t qa = sb + C::kQOff + t * C::kTile;
                const uint32_t kb = sb + C::kKOff + ks * C::kTile;
#pragma unroll
                for (int s = 0; s < D / 16; ++s) {
                    const uint32_t off = (s >> 2) * kBoxBytes + (s & 3) * 32;
                    umma_ss(tmem + C::col_s(t), smem_desc_sw128(qa + off, 16, 1024),
                            smem_desc_sw128(kb + off, 16, 1024), idesc_qk, s > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int t, int vs, bool acc) {
                const uint32_t vb = sb + C::kVOff + vs * C::kTile;
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    umma_ts(tmem + C::col_o(t), tmem + C::col_s(t) + 8 * s,
                            smem_desc_sw128(vb + s * 2048, kBoxBytes, 1024), idesc_pv, (acc || s > 0) ? 1u : 0u);
            };
            mbar_wait(bar(C::kBarQReady), 0, p.wait);
            mbar_wait(bar(C::kBarKReady + 0), 0, p.wait);
            tc_fence_after();
            issue_qk(0, 0);
            tc_commit(bar(C::kBarSFull + 0));
            issue_qk(1, 0);
            tc_commit(bar(C::kBarSFull + 1));
            tc_commit(bar(C::kBarKEmpty + 0));
            for (int j = 0; j < n_kt; ++j) {
                const bool nxt = j + 1 < n_kt;
                const int ks = (j + 1) % kKStages, vs = j % kVStages;
                if (nxt) mbar_wait(bar(C::kBarKReady + ks), ((j + 1) / kKStages) & 1, p.wait);
                mbar_wait(bar(C::kBarVFull + vs), (j / kVStages) & 1, p.wait);
                mbar_wait(bar(C::kBarPReady + 0), j & 1, p.wait);
                tc_fence_after();
                issue_pv(0, vs, j > 0);
                if (nxt) {
                    issue_qk(0, ks);
                    tc_commit(bar(C::kBarSFull + 0));
                } else {
                    tc_commit(bar(C::kBarODone + 0));
                }
                mbar_wait(bar(C::kBarPReady + 1), j & 1, p.wait);
                tc_fence_after();
                issue_pv(1, vs, j > 0);
                tc_commit(bar(C::kBarVEmpty + vs));
                if (nxt) {
                    issue_qk(1, ks);
                    tc_commit(bar(C::kBarSFull + 1));
                    tc_commit(bar(C::kBarKEmpty + ks));
                } else {
                    tc_commit(bar(C::kBarODone + 1));
                }
            }
        }
    } else if (warp >= kWarpRope) {
        // ------------------------------------------------------------ RoPE warps
        const int rt = threadIdx.x - kWarpRope * 32;
        mbar_wait(bar(C::kBarQFull + 0), 0, p.wait);
        mbar_wait(bar(C::kBarQFull + 1), 0, p.wait);
        for (int t = 0; t < 2; ++t) {
            rope_tile<D>(smem + C::kQOff + t * C::kTile, rt, p.rope.cs, [&](int row) {
                const int r = r0 + t * P + row % P;
                return r < p.S_q ? p.q_pos0 + r : -1;
            });
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::kBarQReady));
        for (int j = 0; j < n_kt; ++j) {
            const int ks = j % kKStages;
            const int key0 = 128 * (j_lo + j);
            mbar_wait(bar(C::kBarKFull + ks), (j / kKStages) & 1, p.wait);
            rope_tile<D>(smem + C::kKOff + ks * C::kTile, rt, p.rope.cs, [&](int row) {
                const int key = key0 + row;
                return key < p.S_k ? key : -1;
            });
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kBarKReady + ks));
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int t = warp >> 2;
        const int i = (warp & 3) * 32 + lane;  // row of the M tile == TMEM lane
        const int r = r0 + t * P + i % P;      // query row index
        const int m = p.q_pos0 + r;            // its position
        const int W = p.window;
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t s_addr = lane_base + C::col_s(t);
        const uint32_t o_addr = lane_base + C::col_o(t);
        float m_run = -INFINITY, l_run = 0.f;

        for (int j = 0; j < n_kt; ++j) {
            mbar_wait(bar(C::kBarSFull + t), j & 1, p.wait);
            tc_fence_after();
            const int kstart = 128 * (j_lo + j);
            const bool full_vis = (kstart + 127 <= m) && (W == 0 || m - kstart < W);
            const bool all_full = __all_sync(0xffffffffu, full_vis);

            // pass 1: row max of the visible scores
            float mx = -INFINITY;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t v[32];
                tmem_ld32(s_addr + 32 * ch, v);
                tmem_wait_ld();
                if (all_full) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(v[e]));
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int key = kstart + 32 * ch + e;
                        const bool vis = key <= m && (W == 0 || m - key < W);
                        if (vis) mx = fmaxf(mx, __uint_as_float(v[e]));
                    }
                }
            }
            const float m_tile = mx * p.scale_log2;
            const float m_new = fmaxf(m_run, m_tile);
            const bool need = (m_run != -INFINITY) && (m_new > m_run + 8.f);
            if (__any_sync(0xffffffffu, need)) {
                // raise the reference max of every row of this warp and rescale O and l
                const float alpha = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run - m_new);
                l_run *= alpha;
                m_run = m_new;
#pragma unroll
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t v[32];
                    tmem_ld32(o_addr + 32 * ch, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                    tmem_st32(o_addr + 32 * ch, v);
                }
            } else if (m_run == -INFINITY) {
                m_run = m_new;
            }
            const float m_use = (m_run == -INFINITY) ? 0.f : m_run;

            // pass 2: p = exp2(s * log2(e)/sqrt(d) - m), row sum, P -> TMEM as bf16
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t v[32];
                tmem_ld32(s_addr + 32 * ch, v);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int e2 = 0; e2 < 16; ++e2) {
                    float p0 = fast_exp2(fmaf(__uint_as_float(v[2 * e2]), p.scale_log2, -m_use));
                    float p1 = fast_exp2(fmaf(__uint_as_float(v[2 * e2 + 1]), p.scale_log2, -m_use));
                    if (!all_full) {
                        const int key = kstart + 32 * ch + 2 * e2;
                        if (!(key <= m && (W == 0 || m - key < W))) p0 = 0.f;
                        if (!(key + 1 <= m && (W == 0 || m - key - 1 < W))) p1 = 0.f;
                    }
                    l_run += p0 + p1;
                    pk[e2] = pack_bf16x2(p0, p1);
                }
                tmem_st16(s_addr + 16 * ch, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kBarPReady + t));
        }

        // ---- epilogue: O / l -> bf16 -> shared (TMA box layout) -> TMA store
        mbar_wait(bar(C::kBarODone + t), 0, p.wait);
        tc_fence_after();
        const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
        uint8_t *stile = smem + C::kQOff + t * C::kTile;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t v[32];
            tmem_ld32(o_addr + 32 * ch, v);
            tmem_wait_ld();
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
                w[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * inv, __uint_as_float(v[2 * e + 1]) * inv);
            const int bx = (32 * ch) / 64, c0 = ((32 * ch) % 64) / 8;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
                *reinterpret_cast<uint4 *>(stile + bx * kBoxBytes + swz128(i, c0 + q4)) =
                    make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
        }
        fence_proxy_async_smem();
        named_bar_sync(1 + t, 128);
        if (i == 0 && r0 + t * P < p.S_q) {
#pragma unroll
            for (int bx = 0; bx < C::kBoxes; ++bx)
                tma_store_3d(&tm_o, sb + C::kQOff + t * C::kTile + bx * kBoxBytes, 64 * bx, r0 + t * P, zq);
            bulk_commit_group();
            bulk_wait_group_read0();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D>
cudaError_t launch_t(const PrefillLaunch &L, cudaStream_t stream)
{
    using C = Cfg<D>;
    cudaError_t err =
        cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (err != cudaSuccess) return err;
    prefill_kernel<D><<<L.grid, kThreads, C::kSmemBytes, stream>>>(L.tm_q, L.tm_k, L.tm_v, L.tm_o, L.p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillLaunch &L, cudaStream_t stream)
{
    if (L.p.d_h == 128) return launch_t<128>(L, stream);
    if (L.p.d_h == 64) return launch_t<64>(L, stream);
    return cudaErrorInvalidValue;
}

}  // namespace apex
