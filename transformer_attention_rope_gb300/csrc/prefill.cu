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

constexpr int kThreads = 16 * 32;
// Register split (setmaxnreg): the block is launched with kLaunchRegs per
// thread (512 x 128 = 65536); the softmax warpgroups take kRegsSoftmax, the
// RoPE warpgroup kRegsRope and the producer/MMA warpgroup kRegsCtl.  The host
// refuses to launch unless 128 x (2 kRegsSoftmax + kRegsRope + kRegsCtl) fits
// in what the block was actually launched with.
constexpr int kLaunchRegs = 128;
constexpr int kRegsSoftmax = 176;
constexpr int kRegsRope = 80;
constexpr int kRegsCtl = 80;
static_assert(128 * (2 * kRegsSoftmax + kRegsRope + kRegsCtl) <= kThreads * kLaunchRegs, "register split");
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
    static constexpr int kBarQReady = 2;                      // [2]
    static constexpr int kBarQEmpty = 4;                      // [2]
    static constexpr int kBarKFull = 6;                       // [kKStages]
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

// ---------------------------------------------------------------- RoPE in shared memory
// Tiles are 128 rows x D bf16 stored as D/64 boxes of [128 rows][64 dims] with
// the 128-byte swizzle of the TMA load.  A 16-byte chunk holds 4 interleaved
// pairs (Part 1, §4.2): chunk c of box bx holds pairs 32 bx + 4 c + e, e < 4.

// Rotate the 4 pairs of one chunk, (x_2i, x_2i+1) -> (x c - y s, x s + y c),
// with the angles' (cos, sin) as packed pairs: C[h] = (c_{2h}, c_{2h+1}), etc.
__device__ __forceinline__ uint4 rope_chunk(uint4 v, const uint64_t (&C)[2], const uint64_t (&S)[2])
{
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t w0 = w[2 * h], w1 = w[2 * h + 1];
        const uint64_t X = f2_pack(bf16lo_to_f32(w0), bf16lo_to_f32(w1));  // even elements
        const uint64_t Y = f2_pack(bf16hi_to_f32(w0), bf16hi_to_f32(w1));  // odd elements
        const uint64_t Xn = f2_fma(Y, f2_neg(S[h]), f2_mul(X, C[h]));
        const uint64_t Yn = f2_fma(X, S[h], f2_mul(Y, C[h]));
        float x0, x1, y0, y1;
        f2_unpack(Xn, x0, x1);
        f2_unpack(Yn, y0, y1);
        w[2 * h] = pack_bf16x2(x0, y0);
        w[2 * h + 1] = pack_bf16x2(x1, y1);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// K tile, key row r at position key0 + r.  Thread rt owns chunk c = rt & 7 of
// rows r0 + 16 k (r0 = rt >> 3, k < 8) in every box.  The angles of successive
// rows advance by 16 positions, so (cos, sin) follow the recurrence
// z_{k+1} = z_k * w with w = (cos 16 theta, sin 16 theta), seeded once per tile
// from the table at position key0 + r0.
template <int D>
struct KRope {
    static constexpr int NB = D / 64;
    uint64_t WC[NB][2], WS[NB][2];  // step rotation per pair
    float4 seed[NB][2];             // (c0, s0, c1, s1), (c2, s2, c3, s3) at the tile's first row

    __device__ __forceinline__ void init(const float2 *table, int c)
    {
#pragma unroll
        for (int bx = 0; bx < NB; ++bx) {
            const float4 *p = reinterpret_cast<const float4 *>(table + 16 * (D / 2) + 32 * bx + 4 * c);
            const float4 a = __ldg(p), b = __ldg(p + 1);
            WC[bx][0] = f2_pack(a.x, a.z);
            WS[bx][0] = f2_pack(a.y, a.w);
            WC[bx][1] = f2_pack(b.x, b.z);
            WS[bx][1] = f2_pack(b.y, b.w);
        }
    }
    __device__ __forceinline__ void load_seed(const float2 *table, int pos, int c)
    {
#pragma unroll
        for (int bx = 0; bx < NB; ++bx) {
            const float4 *p = reinterpret_cast<const float4 *>(table + (size_t)pos * (D / 2) + 32 * bx + 4 * c);
            seed[bx][0] = __ldg(p);
            seed[bx][1] = __ldg(p + 1);
        }
    }
    // rotate the tile; reads the seed (the caller may then load the next one)
    __device__ __forceinline__ void rotate(uint8_t *tile, int rt)
    {
        const int c = rt & 7, r0 = rt >> 3;
        uint64_t C[NB][2], S[NB][2];
#pragma unroll
        for (int bx = 0; bx < NB; ++bx) {
            C[bx][0] = f2_pack(seed[bx][0].x, seed[bx][0].z);
            S[bx][0] = f2_pack(seed[bx][0].y, seed[bx][0].w);
            C[bx][1] = f2_pack(seed[bx][1].x, seed[bx][1].z);
            S[bx][1] = f2_pack(seed[bx][1].y, seed[bx][1].w);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int row = r0 + 16 * k;
#pragma unroll
            for (int bx = 0; bx < NB; ++bx) {
                uint4 *ptr = reinterpret_cast<uint4 *>(tile + bx * kBoxBytes + swz128(row, c));
                *ptr = rope_chunk(*ptr, C[bx], S[bx]);
                if (k < 7) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint64_t Cn = f2_fma(C[bx][h], WC[bx][h], f2_mul(S[bx][h], f2_neg(WS[bx][h])));
                        const uint64_t Sn = f2_fma(C[bx][h], WS[bx][h], f2_mul(S[bx][h], WC[bx][h]));
                        C[bx][h] = Cn;
                        S[bx][h] = Sn;
                    }
                }
            }
        }
    }
};

// Q tile: rows are head-major (row = head * P + p), so all G heads of one
// position p share one set of angles.  Thread rt takes the (p, chunk) combos
// rt, rt + 128, ... and rotates that chunk of the G rows of position p.
template <int D>
__device__ __forceinline__ void rope_q_tile(uint8_t *tile, int rt, const float2 *table, int pos0, int G, int P,
                                            int valid_p)
{
    constexpr int NB = D / 64;
    for (int q = rt; q < P * 8; q += 128) {
        const int p = q >> 3, c = q & 7;
        if (p >= valid_p) continue;
        uint64_t C[NB][2], S[NB][2];
#pragma unroll
        for (int bx = 0; bx < NB; ++bx) {
            const float4 *t = reinterpret_cast<const float4 *>(table + (size_t)(pos0 + p) * (D / 2) + 32 * bx + 4 * c);
            const float4 a = __ldg(t), b = __ldg(t + 1);
            C[bx][0] = f2_pack(a.x, a.z);
            S[bx][0] = f2_pack(a.y, a.w);
            C[bx][1] = f2_pack(b.x, b.z);
            S[bx][1] = f2_pack(b.y, b.w);
        }
        for (int hl = 0; hl < G; ++hl) {
            const int row = hl * P + p;
#pragma unroll
            for (int bx = 0; bx < NB; ++bx) {
                uint4 *ptr = reinterpret_cast<uint4 *>(tile + bx * kBoxBytes + swz128(row, c));
                *ptr = rope_chunk(*ptr, C[bx], S[bx]);
            }
        }
    }
}

// One work item: (batch, kv head) unit and a block of 2P query rows.
struct Item {
    int unit, b, hk, r0, j_lo, n_kt, zq;
};

__device__ __forceinline__ Item make_item(const PrefillParams &p, int w)
{
    Item it;
    const int units = p.B * p.H_kv;
    const int qblock = p.n_qblocks - 1 - w / units;  // latest positions (most key tiles) first
    it.unit = w % units;
    it.b = it.unit / p.H_kv;
    it.hk = it.unit % p.H_kv;
    const int P = p.rows_per_head;
    it.r0 = qblock * 2 * P;
    const int rows = min(2 * P, p.S_q - it.r0);
    const int m_first = p.q_pos0 + it.r0, m_last = p.q_pos0 + it.r0 + rows - 1;
    // union of the rows' visible key ranges: [lo(m), m] (Part 2, §10.2), or the
    // whole prefix [0, P) for rows inside it (§11.1)
    const int key_lo = (m_first < p.prefix_len || p.window <= 0) ? 0 : max(0, m_first - p.window + 1);
    const int key_hi = (m_first < p.prefix_len) ? max(m_last, p.prefix_len - 1) : m_last;
    it.j_lo = key_lo / 128;
    it.n_kt = key_hi / 128 - it.j_lo + 1;
    it.zq = it.b * p.H_q + it.hk * p.G;
    return it;
}

// k-th item of this CTA: rounds of gridDim.x items, walked in alternating
// direction so that the heavy items of each round spread over the CTAs.
__device__ __forceinline__ int item_index(int k)
{
    const int g = gridDim.x, c = blockIdx.x;
    return k * g + ((k & 1) ? (g - 1 - c) : c);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillParams p)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) -> uint32_t { return sb + C::kBarOff + 8 * i; };
    const int P = p.rows_per_head;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(C::kBarQFull + t), 1);
            mbar_init(bar(C::kBarQReady + t), 4);
            mbar_init(bar(C::kBarQEmpty + t), 1);
            mbar_init(bar(C::kBarSFull + t), 1);
            mbar_init(bar(C::kBarPReady + t), 4);
            mbar_init(bar(C::kBarODone + t), 1);
        }
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(bar(C::kBarKFull + s), 1);
            mbar_init(bar(C::kBarKReady + s), 4);
            mbar_init(bar(C::kBarKEmpty + s), 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(bar(C::kBarVFull + s), 1);
            mbar_init(bar(C::kBarVEmpty + s), 1);
        }
        fence_mbarrier_init();
    }
    if (warp == kWarpMma) tmem_alloc(sb + C::kTmemSlot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + C::kTmemSlot);
    // launched as a programmatic dependent: the set-up above overlaps the previous
    // kernel's tail; nothing in global memory is touched before that kernel is done
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp >= kWarpTma) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
    if (warp == kWarpTma) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            int kc = 0;  // K/V tiles issued so far (ring position)
            for (int k = 0, w = item_index(0); w < p.n_work; ++k, w = item_index(k)) {
                const Item it = make_item(p, w);
                for (int t = 0; t < 2; ++t) {
                    mbar_wait(bar(C::kBarQEmpty + t), (k & 1) ^ 1, p.wait);
                    mbar_arrive_expect_tx(bar(C::kBarQFull + t), C::kTile);
#pragma unroll
                    for (int bx = 0; bx < C::kBoxes; ++bx)
                        tma_load_3d(sb + C::kQOff + t * C::kTile + bx * kBoxBytes, &tm_q, bar(C::kBarQFull + t),
                                    64 * bx, it.r0 + t * P, it.zq);
                }
                for (int j = 0; j < it.n_kt; ++j, ++kc) {
                    const int key0 = 128 * (it.j_lo + j);
                    const int ks = kc % kKStages, vs = kc % kVStages;
                    mbar_wait(bar(C::kBarKEmpty + ks), ((kc / kKStages) & 1) ^ 1, p.wait);
                    mbar_arrive_expect_tx(bar(C::kBarKFull + ks), C::kTile);
#pragma unroll
                    for (int bx = 0; bx < C::kBoxes; ++bx)
                        tma_load_3d(sb + C::kKOff + ks * C::kTile + bx * kBoxBytes, &tm_k, bar(C::kBarKFull + ks),
                                    64 * bx, key0, it.unit);
                    mbar_wait(bar(C::kBarVEmpty + vs), ((kc / kVStages) & 1) ^ 1, p.wait);
                    mbar_arrive_expect_tx(bar(C::kBarVFull + vs), C::kTile);
#pragma unroll
                    for (int bx = 0; bx < C::kBoxes; ++bx)
                        tma_load_3d(sb + C::kVOff + vs * C::kTile + bx * kBoxBytes, &tm_v, bar(C::kBarVFull + vs),
                                    64 * bx, key0, it.unit);
                }
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
            // One descriptor per operand and call, stepped by adding the k-step's
            // offset (>> 4) to its address field; the empty asm keeps the base a
            // runtime value, so the compiler does not precompute (and keep live)
            // the descriptors of every tile and stage.
            auto desc_base = [&](uint32_t addr, uint32_t lbo) -> uint64_t {
                uint64_t d = smem_desc_sw128(addr, lbo, 1024);
                asm volatile("" : "+l"(d));
                return d;
            };
            auto issue_qk = [&](int t, int ks) {
                const uint64_t da = desc_base(sb + C::kQOff + t * C::kTile, 16);
                const uint64_t db = desc_base(sb + C::kKOff + ks * C::kTile, 16);
#pragma unroll
                for (int s = 0; s < D / 16; ++s) {
                    const uint64_t off = ((s >> 2) * kBoxBytes + (s & 3) * 32) >> 4;
                    umma_ss(tmem + C::col_s(t), da + off, db + off, idesc_qk, s > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int t, int vs, bool acc) {
                const uint64_t dv = desc_base(sb + C::kVOff + vs * C::kTile, kBoxBytes);
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    umma_ts(tmem + C::col_o(t), tmem + C::col_s(t) + 8 * s, dv + (uint64_t)(s * 2048 >> 4), idesc_pv,
                            (acc || s > 0) ? 1u : 0u);
            };
            int kc = 0;
            for (int k = 0, w = item_index(0); w < p.n_work; ++k, w = item_index(k)) {
                const Item it = make_item(p, w);
                const int n = it.n_kt;
                mbar_wait(bar(C::kBarKReady + kc % kKStages), (kc / kKStages) & 1, p.wait);
                for (int t = 0; t < 2; ++t) {
                    mbar_wait(bar(C::kBarQReady + t), k & 1, p.wait);
                    tc_fence_after();
                    issue_qk(t, kc % kKStages);
                    tc_commit(bar(C::kBarSFull + t));
                    if (n == 1) tc_commit(bar(C::kBarQEmpty + t));  // last read of Q_t
                }
                tc_commit(bar(C::kBarKEmpty + kc % kKStages));
                for (int j = 0; j < n; ++j) {
                    const int g = kc + j;
                    const bool nxt = j + 1 < n;
                    const bool last_qk = j + 2 == n;  // the next QK is this item's last read of Q
                    const int ks = (g + 1) % kKStages, vs = g % kVStages;
                    mbar_wait(bar(C::kBarVFull + vs), (g / kVStages) & 1, p.wait);
                    mbar_wait(bar(C::kBarPReady + 0), g & 1, p.wait);
                    tc_fence_after();
                    issue_pv(0, vs, j > 0);
                    if (nxt) {
                        mbar_wait(bar(C::kBarKReady + ks), ((g + 1) / kKStages) & 1, p.wait);
                        tc_fence_after();
                        issue_qk(0, ks);
                        tc_commit(bar(C::kBarSFull + 0));
                        if (last_qk) tc_commit(bar(C::kBarQEmpty + 0));
                    } else {
                        tc_commit(bar(C::kBarODone + 0));
                    }
                    mbar_wait(bar(C::kBarPReady + 1), g & 1, p.wait);
                    tc_fence_after();
                    issue_pv(1, vs, j > 0);
                    tc_commit(bar(C::kBarVEmpty + vs));
                    if (nxt) {
                        issue_qk(1, ks);
                        tc_commit(bar(C::kBarSFull + 1));
                        if (last_qk) tc_commit(bar(C::kBarQEmpty + 1));
                        tc_commit(bar(C::kBarKEmpty + ks));
                    } else {
                        tc_commit(bar(C::kBarODone + 1));
                    }
                }
                kc += n;
            }
        }
    } else if (warp >= kWarpRope && warp < kWarpTma) {
        // ------------------------------------------------------------ RoPE warps
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsRope));
        const int rt = threadIdx.x - kWarpRope * 32;
        const int c = rt & 7, r0 = rt >> 3;
        const int max_row = p.rope.max_pos - 1;
        KRope<D> kr;
        kr.init(p.rope.cs, c);
        int kc = 0;
        for (int k = 0, w = item_index(0); w < p.n_work; ++k, w = item_index(k)) {
            const Item it = make_item(p, w);
            kr.load_seed(p.rope.cs, min(128 * it.j_lo + r0, max_row), c);
            for (int j = 0; j < it.n_kt; ++j, ++kc) {
                const int ks = kc % kKStages;
                mbar_wait(bar(C::kBarKFull + ks), (kc / kKStages) & 1, p.wait);
                if (!p.keys_prerotated) kr.rotate(smem + C::kKOff + ks * C::kTile, rt);
                if (j + 1 < it.n_kt) kr.load_seed(p.rope.cs, min(128 * (it.j_lo + j + 1) + r0, max_row), c);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::kBarKReady + ks));
            }
        }
    } else if (warp < kWarpRope) {
        // ------------------------------------------------------------ softmax + epilogue
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        const int t = warp >> 2;
        const int i = (warp & 3) * 32 + lane;  // row of the M tile == TMEM lane
        const int W = p.window;
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t s_addr = lane_base + C::col_s(t);
        const uint32_t o_addr = lane_base + C::col_o(t);
        // RoPE of this warpgroup's Q tile of an item (rows at or past S_q are padding)
        auto rotate_q = [&](const Item &it, int k) {
            mbar_wait(bar(C::kBarQFull + t), k & 1, p.wait);
            rope_q_tile<D>(smem + C::kQOff + t * C::kTile, i, p.rope.cs, p.q_pos0 + it.r0 + t * P, p.G, P,
                           min(P, p.S_q - (it.r0 + t * P)));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::kBarQReady + t));
        };
        int kc = 0;
        if (item_index(0) < p.n_work) rotate_q(make_item(p, item_index(0)), 0);
        for (int k = 0, w = item_index(0); w < p.n_work; ++k, w = item_index(k)) {
            const Item it = make_item(p, w);
            const int r = it.r0 + t * P + i % P;  // query row index
            const int m = p.q_pos0 + r;           // its position
            // keys this row sees: [key_lo, key_hi]
            const bool in_prefix = m < p.prefix_len;
            const int key_lo = (in_prefix || W <= 0) ? 0 : m - W + 1;
            const int key_hi = in_prefix ? p.prefix_len - 1 : m;
            float m_run = -INFINITY, l_run = 0.f;

            for (int j = 0; j < it.n_kt; ++j) {
                mbar_wait(bar(C::kBarSFull + t), (kc + j) & 1, p.wait);
                tc_fence_after();
                const int kstart = 128 * (it.j_lo + j);
                // columns [lo_c, hi_c] of this tile are visible to the row
                const int hi_c = key_hi - kstart;
                const int lo_c = key_lo - kstart;
                const bool full_vis = lo_c <= 0 && hi_c >= 127;
                const bool all_full = __all_sync(0xffffffffu, full_vis);
                // the whole 128-column row of S in registers
                uint32_t v[128];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    tmem_ld32(s_addr + 32 * ch, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * ch]));
                tmem_wait_ld();
                if (!all_full) mask_row128(v, lo_c, hi_c);
                // row max of the visible scores (8 independent chains)
                float acc[8];
#pragma unroll
                for (int a = 0; a < 8; ++a) acc[a] = __uint_as_float(v[a]);
#pragma unroll
                for (int e = 8; e + 16 <= 128; e += 16)  // columns 8 .. 119
#pragma unroll
                    for (int a = 0; a < 8; ++a)
                        acc[a] = fmax3(acc[a], __uint_as_float(v[e + a]), __uint_as_float(v[e + 8 + a]));
#pragma unroll
                for (int a = 0; a < 8; ++a) acc[a] = fmaxf(acc[a], __uint_as_float(v[120 + a]));
                const float mx = fmax3(fmax3(acc[0], acc[1], acc[2]), fmax3(acc[3], acc[4], acc[5]), fmaxf(acc[6], acc[7]));
                const float m_tile = mx * p.scale_log2;
                const float m_new = fmaxf(m_run, m_tile);
                const bool need = (m_run != -INFINITY) && (m_new > m_run + 8.f);
                if (__any_sync(0xffffffffu, need)) {
                    // raise the reference max of every row of this warp and rescale O and l
                    const float alpha = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run - m_new);
                    l_run *= alpha;
                    m_run = m_new;
#pragma unroll 1
                    for (int ch = 0; ch < D / 16; ++ch) {
                        uint32_t o[16];
                        tmem_ld16(o_addr + 16 * ch, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st16(o_addr + 16 * ch, o);
                    }
                } else if (m_run == -INFINITY) {
                    m_run = m_new;
                }
                const float m_use = (m_run == -INFINITY) ? 0.f : m_run;

                // p = exp2(s * log2(e)/sqrt(d) - m), row sum, P -> TMEM as bf16 over S
                const uint64_t SC = f2_pack(p.scale_log2, p.scale_log2);
                const uint64_t NM = f2_pack(-m_use, -m_use);
                uint64_t lacc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e2 = 0; e2 < 16; ++e2) {
                        const uint64_t x = f2_pack(__uint_as_float(v[32 * q4 + 2 * e2]), __uint_as_float(v[32 * q4 + 2 * e2 + 1]));
                        float y0, y1;
                        f2_unpack(f2_fma(x, SC, NM), y0, y1);
                        const float p0 = fast_exp2(y0), p1 = fast_exp2(y1);
                        lacc[e2 & 3] = f2_add(lacc[e2 & 3], f2_pack(p0, p1));
                        pk[e2] = pack_bf16x2(p0, p1);
                    }
                    tmem_st16(s_addr + 16 * q4, pk);
                }
                {
                    float a0, a1;
                    f2_unpack(f2_add(f2_add(lacc[0], lacc[1]), f2_add(lacc[2], lacc[3])), a0, a1);
                    l_run += a0 + a1;
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::kBarPReady + t));
            }
            kc += it.n_kt;

            // the next item's Q tile was loaded once this item's last QK was done:
            // rotate it now, so its first QK overlaps this item's epilogue
            const int w_next = item_index(k + 1);
            if (w_next < p.n_work) rotate_q(make_item(p, w_next), k + 1);

            // ---- epilogue: O / l -> bf16 -> global, one row per thread
            mbar_wait(bar(C::kBarODone + t), k & 1, p.wait);
            tc_fence_after();
            const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
            const int hl = i / P;
            uint4 *dst = reinterpret_cast<uint4 *>(p.out + ((size_t)(it.zq + hl) * p.S_q + r) * D);
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t v[32];
                tmem_ld32(o_addr + 32 * ch, v);
                tmem_wait_ld();
                uint32_t w2[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w2[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * inv, __uint_as_float(v[2 * e + 1]) * inv);
                if (r < p.S_q) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        dst[4 * ch + q4] = make_uint4(w2[4 * q4], w2[4 * q4 + 1], w2[4 * q4 + 2], w2[4 * q4 + 3]);
                }
            }
            tc_fence_before();
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
    // setmaxnreg.inc blocks until the block's own pool can serve it: never
    // launch unless the split fits the registers the block is launched with
    cudaFuncAttributes fa;
    err = cudaFuncGetAttributes(&fa, prefill_kernel<D>);
    if (err != cudaSuccess) return err;
    if (fa.numRegs < kLaunchRegs) return cudaErrorInvalidConfiguration;
    return launch_dependent(prefill_kernel<D>, L.grid, kThreads, C::kSmemBytes, stream, L.tm_q, L.tm_k, L.tm_v, L.p);
}

}  // namespace

cudaError_t launch_prefill(const PrefillLaunch &L, cudaStream_t stream)
{
    if (L.p.d_h == 128) return launch_t<128>(L, stream);
    if (L.p.d_h == 64) return launch_t<64>(L, stream);
    return cudaErrorInvalidValue;
}

}  // namespace apex
