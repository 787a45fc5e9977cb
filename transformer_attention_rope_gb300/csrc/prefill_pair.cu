// prefill_pair.cu -- the prefill on CTA pairs (tcgen05 cta_group::2), value and
// output rows of 128 entries; query and key rows of DQK = 128 entries (the
// plain block, RoPE over the whole row) or 192 (multi-head latent attention with
// decoupled RoPE, Part 2, §9.3: rows [content (128) | rope part (64)], RoPE of
// dimension 64 on the rope part only).
//
// Same computation as prefill.cu (RoPE on Q and K tiles in shared memory, GQA
// packing of the G heads that share a KV head into each 128-row M tile, online
// exp2 softmax, key tiles outside the causal/window/prefix bounds skipped), but
// a work item is four M tiles of one (batch, kv head) unit spread over the two
// CTAs of a cluster, and each 128-key tile is shared by both CTAs:
//
//   * S_t = Q_t K^T and O_t += P_t V run as M = 256 MMAs issued by the leader
//     CTA (rank 0): rows 0-127 are the leader's tile t, rows 128-255 the
//     peer's; the B operand is split along N between the two shared memories,
//     so each CTA loads -- and rotates -- only 64 of the 128 keys of every K
//     tile, and holds only 64 of the 128 dims of every V tile.
//   * TMEM is allocated for the pair; each CTA's softmax warpgroups read their
//     own S rows and write their own P and O rows, as in the single-CTA kernel.
//   * The leader's MMA thread waits on its own barriers, which the peer's warps
//     reach through remote (shared::cluster) arrivals; its commits are
//     multicast, so every CTA waits on local barriers only.
//
// Warps per CTA: 0-3 / 4-7 softmax + epilogue of tiles 0 / 1 (and their Q
// RoPE), 8-11 K RoPE (their "K ready" arrival also vouches that the V tile of
// the same index has landed, so the MMA thread has one wait less per tile; in
// the instance for keys rotated beforehand they turn no K tile, and for G >= 8
// rotate a share of the Q tiles instead), 12 TMA producer, 13 MMA issuer
// (leader) / TMEM allocation, 14-15 idle.
#include <math.h>

#include "device_common.cuh"
#include "tcgen05.cuh"

namespace apex {
namespace {

constexpr int DV = 128;  // value / output row length
constexpr int kThreads = 16 * 32;
constexpr int kWarpRope = 8;
constexpr int kWarpTma = 12;
constexpr int kWarpMma = 13;
constexpr int kLaunchRegs = 128;
constexpr int kRegsSoftmax = 176;
constexpr int kRegsRope = 88;
constexpr int kRegsCtl = 72;
static_assert(128 * (2 * kRegsSoftmax + kRegsRope + kRegsCtl) <= kThreads * kLaunchRegs, "register split");

constexpr int kQBox = 128 * 128;  // [128 rows][64 dims]
constexpr int kKBox = 64 * 128;   // [64 keys][64 dims]
constexpr int kVTile = 128 * 128; // 128 keys x this CTA's 64 dims

// DQK: query / key row length; DR: trailing entries of those rows that RoPE turns.
template <int DQK, int DR>
struct PairCfg {
    static_assert(DQK % 64 == 0 && DR % 64 == 0 && DR <= DQK, "row split");
    static constexpr int kBoxes = DQK / 64;          // 64-dim boxes of a Q or K row
    static constexpr int kRopeBox0 = (DQK - DR) / 64; // first box of the rope part
    static constexpr int kRopeBoxes = DR / 64;
    static constexpr int kStages = 3;  // 4 measured 1-2 % slower for 128-wide rows
    static constexpr int kKStages = kStages;
    static constexpr int kVStages = kStages;  // K(x) and V(x) share stage x % kStages and one "empty" barrier
    static constexpr int kQTile = kBoxes * kQBox;     // 128 rows x DQK
    static constexpr int kKTile = kBoxes * kKBox;     // this CTA's 64 keys x DQK
    // O leaves through shared memory and TMA stores where there is room for the
    // staging buffers (128-wide rows); the 192-wide rows keep per-thread stores.
    static constexpr bool kTmaStoreO = DQK == 128;
    static constexpr int kStageWarpBytes = 32 * DV * 2;  // one softmax warp's 32 rows of O, bf16
    // Q | V stages | K stages | O staging (8 softmax warps) or 8 KB guard |
    // barriers: an operand descriptor that walked past its tile (it should not:
    // each CTA's B half is 64 rows or 64 columns) would still stay inside the
    // allocation.
    static constexpr int kQOff = 0;
    static constexpr int kVOff = 2 * kQTile;
    static constexpr int kKOff = kVOff + kVStages * kVTile;
    static constexpr int kStageOff = kKOff + kKStages * kKTile;
    static constexpr int kBarOff = kStageOff + (kTmaStoreO ? 8 * kStageWarpBytes : 8192);
    static_assert(kStageOff % 1024 == 0, "staging buffers need 1024-byte alignment for the 128-byte swizzle");
    // barrier slots
    static constexpr int kBarQFull = 0;                         // [2]  local TMA
    static constexpr int kBarQReady = 2;                        // [2]  leader: 8 warps (both CTAs)
    static constexpr int kBarQEmpty = 4;                        // [2]  multicast commit
    static constexpr int kBarSFull = 6;                         // [2]  multicast commit
    static constexpr int kBarPReady = 8;                        // [2]  leader: 8 warps
    static constexpr int kBarODone = 10;                        // [2]  multicast commit
    static constexpr int kBarKFull = 12;                        // [K]  local TMA
    static constexpr int kBarKReady = kBarKFull + kKStages;     // [K]  leader: 8 warps
    static constexpr int kBarVFull = kBarKReady + kKStages;     // [V]  local TMA
    static constexpr int kBarVEmpty = kBarVFull + kVStages;     // [V]  multicast commit: frees K and V stage
    static constexpr int kNumBars = kBarVEmpty + kVStages;
    static constexpr int kTmemSlot = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kTmemSlot + 16 + 1024;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ uint32_t col_s(int t) { return 128u * t; }
__device__ __forceinline__ uint32_t col_o(int t) { return 256u + 128u * t; }

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// ---------------------------------------------------------------- cluster helpers
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on the barrier at the same shared-memory offset in the leader CTA.
// Default (release, CTA-scope) semantics: a cluster-scope release here costs
// about a microsecond per arrival on the softmax critical path.
__device__ __forceinline__ void arrive_leader(uint32_t local_bar)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_bar), "r"(0));
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}

// Bounded wait on a local barrier (some receive arrivals from the peer CTA).
// On time-out the status word and the CTA's abort flag (shared memory) are
// set and the wait returns; once the flag is set, later waits of the CTA that
// do not complete at once give up at their first timer check, so a broken
// pipeline drains in about one time-out.
__device__ __forceinline__ void pair_wait(uint32_t bar, uint32_t parity, const WaitCtl &wc, volatile uint32_t *abort)
{
    if (mbar_try_wait(bar, parity)) return;
    uint64_t t0 = 0;
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return;
        if ((n & 255u) == 0) {
            if (*abort) return;
            const uint64_t now = global_timer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > wc.timeout_ns) {
                *abort = 1u;
                report_status(wc.status, kStatusWaitTimeout);
                return;
            }
        }
    }
}

__device__ __forceinline__ void commit_pair(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                     bar),
                 "h"((uint16_t)3)
                 : "memory");
}

__device__ __forceinline__ void mma_ss_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// ---------------------------------------------------------------- RoPE in shared memory
// A 16-byte chunk holds 4 interleaved pairs (Part 1, §4.2): chunk c of box bx
// holds pairs 32 bx + 4 c + e, e < 4.  (x_2i, x_2i+1) -> (x c - y s, x s + y c)
// in fp32 on packed pairs, rounded to bf16.
__device__ __forceinline__ uint4 rope_chunk(uint4 v, const uint64_t (&C)[2], const uint64_t (&S)[2])
{
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t w0 = w[2 * h], w1 = w[2 * h + 1];
        const uint64_t X = f2_pack(bf16lo_to_f32(w0), bf16lo_to_f32(w1));
        const uint64_t Y = f2_pack(bf16hi_to_f32(w0), bf16hi_to_f32(w1));
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

// This CTA's half of a K tile: 64 key rows (position pos0 + r), stored as
// 64-dim swizzled boxes of [64 rows][64 dims]; RoPE turns boxes B0 .. B0+NRB-1,
// whose pairs are numbered from the start of the rope part (table rows hold
// DR/2 = 32 NRB pairs).  Thread rt owns chunk c = rt & 7 of rows r0 + 16 k
// (r0 = rt >> 3, k < 4); the angle advances by 16 positions per step:
// z_{k+1} = z_k * (cos 16 theta, sin 16 theta), seeded per tile.
template <int NRB, int B0>
struct KHalfRope {
    static constexpr int kHalf = 32 * NRB;  // pairs per table row
    uint64_t WC[NRB][2], WS[NRB][2];
    float4 seed[NRB][2];

    __device__ __forceinline__ void init(const float2 *table, int c)
    {
#pragma unroll
        for (int bx = 0; bx < NRB; ++bx) {
            const float4 *p = reinterpret_cast<const float4 *>(table + 16 * kHalf + 32 * bx + 4 * c);
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
        for (int bx = 0; bx < NRB; ++bx) {
            const float4 *p = reinterpret_cast<const float4 *>(table + (size_t)pos * kHalf + 32 * bx + 4 * c);
            seed[bx][0] = __ldg(p);
            seed[bx][1] = __ldg(p + 1);
        }
    }
    __device__ __forceinline__ void rotate(uint8_t *tile, int rt)
    {
        const int c = rt & 7, r0 = rt >> 3;
        uint64_t C[NRB][2], S[NRB][2];
#pragma unroll
        for (int bx = 0; bx < NRB; ++bx) {
            C[bx][0] = f2_pack(seed[bx][0].x, seed[bx][0].z);
            S[bx][0] = f2_pack(seed[bx][0].y, seed[bx][0].w);
            C[bx][1] = f2_pack(seed[bx][1].x, seed[bx][1].z);
            S[bx][1] = f2_pack(seed[bx][1].y, seed[bx][1].w);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int row = r0 + 16 * k;
#pragma unroll
            for (int bx = 0; bx < NRB; ++bx) {
                uint4 *ptr = reinterpret_cast<uint4 *>(tile + (B0 + bx) * kKBox + swz128(row, c));
                *ptr = rope_chunk(*ptr, C[bx], S[bx]);
                if (k < 3) {
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

// Q tile: head-major rows (row = head * P + p); all G heads of position p share
// one set of angles.  Thread rt takes the (p, chunk) combos rt, rt + 128, ...
// and turns boxes B0 .. B0+NRB-1 (the rope part) of that chunk.
template <int NRB, int B0>
__device__ __forceinline__ void rope_q_tile(uint8_t *tile, int rt, const float2 *table, int pos0, int G, int P,
                                            int valid_p)
{
    constexpr int kHalf = 32 * NRB;
    for (int q = rt; q < P * 8; q += 128) {
        const int pp = q >> 3, c = q & 7;
        if (pp >= valid_p) continue;
        uint64_t C[NRB][2], S[NRB][2];
#pragma unroll
        for (int bx = 0; bx < NRB; ++bx) {
            const float4 *t = reinterpret_cast<const float4 *>(table + (size_t)(pos0 + pp) * kHalf + 32 * bx + 4 * c);
            const float4 a = __ldg(t), b = __ldg(t + 1);
            C[bx][0] = f2_pack(a.x, a.z);
            S[bx][0] = f2_pack(a.y, a.w);
            C[bx][1] = f2_pack(b.x, b.z);
            S[bx][1] = f2_pack(b.y, b.w);
        }
        for (int hl = 0; hl < G; ++hl) {
            const int row = hl * P + pp;
#pragma unroll
            for (int bx = 0; bx < NRB; ++bx) {
                uint4 *ptr = reinterpret_cast<uint4 *>(tile + (B0 + bx) * kQBox + swz128(row, c));
                *ptr = rope_chunk(*ptr, C[bx], S[bx]);
            }
        }
    }
}

// Part of a Q tile: combos q = q_first, q_first + q_step, ... (< 8P) of position
// q >> 3 and chunk q & 7, heads [h_lo, h_hi) of each.
template <int NRB, int B0>
__device__ __forceinline__ void rope_q_part(uint8_t *tile, const float2 *table, int pos0, int P, int valid_p,
                                            int q_first, int q_step, int h_lo, int h_hi)
{
    constexpr int kHalf = 32 * NRB;
    for (int q = q_first; q < P * 8; q += q_step) {
        const int pp = q >> 3, c = q & 7;
        if (pp >= valid_p) continue;
        uint64_t C[NRB][2], S[NRB][2];
#pragma unroll
        for (int bx = 0; bx < NRB; ++bx) {
            const float4 *t = reinterpret_cast<const float4 *>(table + (size_t)(pos0 + pp) * kHalf + 32 * bx + 4 * c);
            const float4 a = __ldg(t), b = __ldg(t + 1);
            C[bx][0] = f2_pack(a.x, a.z);
            S[bx][0] = f2_pack(a.y, a.w);
            C[bx][1] = f2_pack(b.x, b.z);
            S[bx][1] = f2_pack(b.y, b.w);
        }
        for (int hl = h_lo; hl < h_hi; ++hl) {
            const int row = hl * P + pp;
#pragma unroll
            for (int bx = 0; bx < NRB; ++bx) {
                uint4 *ptr = reinterpret_cast<uint4 *>(tile + (B0 + bx) * kQBox + swz128(row, c));
                *ptr = rope_chunk(*ptr, C[bx], S[bx]);
            }
        }
    }
}

// With the keys rotated beforehand (the K-RoPE warps have no K tiles to turn)
// and G >= 8, the K-RoPE warps rotate the last G / 4 heads of both Q tiles of
// each item, the softmax warps the others: per thread 6 (position, head) pairs
// instead of 8 (G = 8) or 16 (G = 16, where only 64 positions x 8 chunks exist
// for 128 threads).  Measured: G = 16 3.5 % faster; at G = 4, where the softmax
// warps' share only drops from 8 to 6, it is not faster.
__device__ __forceinline__ bool q_shared(bool krot, int G) { return !krot && G >= 8; }
__device__ __forceinline__ int q_heads_softmax(int G) { return G - G / 4; }

// ---------------------------------------------------------------- work items
// One item: a (batch, kv head) unit and a block of 4P query rows (P = 128 / G):
// tile T = 2 rank + t of the pair covers rows r0 + T P .. r0 + T P + P - 1.
struct Item {
    int unit, r0, j_lo, n_kt, zq;
};

__device__ __forceinline__ Item make_item(const PrefillParams &p, int w)
{
    Item it;
    const int units = p.B * p.H_kv;
    const int qblock = p.n_qblocks - 1 - w / units;  // latest positions (most key tiles) first
    it.unit = w % units;
    const int b = it.unit / p.H_kv, hk = it.unit % p.H_kv;
    const int P = p.rows_per_head;
    it.r0 = qblock * 4 * P;
    const int rows = min(4 * P, p.S_q - it.r0);
    const int m_first = p.q_pos0 + it.r0, m_last = p.q_pos0 + it.r0 + rows - 1;
    const int key_lo = (m_first < p.prefix_len || p.window <= 0) ? 0 : max(0, m_first - p.window + 1);
    const int key_hi = (m_first < p.prefix_len) ? max(m_last, p.prefix_len - 1) : m_last;
    it.j_lo = key_lo / 128;
    it.n_kt = key_hi / 128 - it.j_lo + 1;
    it.zq = b * p.H_q + hk * p.G;
    return it;
}

// k-th item of this pair: rounds of n_pairs items, walked in alternating direction.
__device__ __forceinline__ int item_index(int k)
{
    const int g = gridDim.x >> 1, c = blockIdx.x >> 1;
    return k * g + ((k & 1) ? (g - 1 - c) : c);
}

// KROT: the K tiles are rotated in shared memory; false: the instance for keys
// rotated beforehand (by the library's key pass or by the caller), at both row
// widths.
template <int DQK, int DR, bool KROT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                        const PrefillParams p)
{
    using C = PairCfg<DQK, DR>;
    constexpr int kKStages = C::kKStages, kVStages = C::kVStages;
    constexpr int kQTile = C::kQTile, kKTile = C::kKTile;
    constexpr int kQOff = C::kQOff, kKOff = C::kKOff, kVOff = C::kVOff, kBarOff = C::kBarOff;
    constexpr int kTmemSlot = C::kTmemSlot;
    constexpr int kBarQFull = C::kBarQFull, kBarQReady = C::kBarQReady, kBarQEmpty = C::kBarQEmpty;
    constexpr int kBarSFull = C::kBarSFull, kBarPReady = C::kBarPReady, kBarODone = C::kBarODone;
    constexpr int kBarKFull = C::kBarKFull, kBarKReady = C::kBarKReady;
    constexpr int kBarVFull = C::kBarVFull, kBarVEmpty = C::kBarVEmpty;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    auto bar = [&](int i) -> uint32_t { return sb + kBarOff + 8 * i; };
    const int P = p.rows_per_head;
    volatile uint32_t *abort = reinterpret_cast<volatile uint32_t *>(smem + kTmemSlot + 4);

    if (threadIdx.x == 0) {
        *abort = 0u;
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(kBarQFull + t), 1);
            mbar_init(bar(kBarQReady + t), q_shared(KROT, p.G) ? 16 : 8);
            mbar_init(bar(kBarQEmpty + t), 1);
            mbar_init(bar(kBarSFull + t), 1);
            mbar_init(bar(kBarPReady + t), 8);
            mbar_init(bar(kBarODone + t), 1);
        }
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(bar(kBarKFull + s), 1);
            mbar_init(bar(kBarKReady + s), 8);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(bar(kBarVFull + s), 1);
            mbar_init(bar(kBarVEmpty + s), 1);
        }
        fence_mbarrier_init();
    }
    if (warp == kWarpMma) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sb + kTmemSlot),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + kTmemSlot);
    // launched as a programmatic dependent: the set-up above overlaps the previous
    // kernel's tail; nothing in global memory is touched before that kernel is done
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp >= kWarpTma) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
    if (warp == kWarpTma) {
        // ------------------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            if (C::kTmaStoreO) tma_prefetch_desc(&tm_o);
            int kc = 0;
            for (int k = 0, w = item_index(0); w < p.n_work; ++k, w = item_index(k)) {
                const Item it = make_item(p, w);
                auto load_q = [&]() {
                    for (int t = 0; t < 2; ++t) {
                        pair_wait(bar(kBarQEmpty + t), (k & 1) ^ 1, p.wait, abort);
                        mbar_arrive_expect_tx(bar(kBarQFull + t), kQTile);
#pragma unroll
                        for (int bx = 0; bx < C::kBoxes; ++bx)
                            tma_load_3d(sb + kQOff + t * kQTile + bx * kQBox, &tm_q, bar(kBarQFull + t), 64 * bx,
                                        it.r0 + (2 * (int)rank + t) * P, it.zq);
                    }
                };
                for (int j = 0; j < it.n_kt; ++j, ++kc) {
                    const int key0 = 128 * (it.j_lo + j);
                    const int ks = kc % kKStages, vs = kc % kVStages;
                    // one "stage empty" barrier frees K(kc) and V(kc) together: it is
                    // committed after PV(kc - stages), which follows QK(kc - stages)
                    pair_wait(bar(kBarVEmpty + vs), ((kc / kVStages) & 1) ^ 1, p.wait, abort);
                    mbar_arrive_expect_tx(bar(kBarKFull + ks), kKTile);
#pragma unroll
                    for (int bx = 0; bx < C::kBoxes; ++bx)
                        tma_load_3d(sb + kKOff + ks * kKTile + bx * kKBox, &tm_k, bar(kBarKFull + ks), 64 * bx,
                                    key0 + 64 * (int)rank, it.unit);
                    mbar_arrive_expect_tx(bar(kBarVFull + vs), kVTile);
                    tma_load_3d(sb + kVOff + vs * kVTile, &tm_v, bar(kBarVFull + vs), 64 * (int)rank, key0, it.unit);
                    // the item's first K / V tiles go out before its Q tiles, whose
                    // buffers free up only when the previous item's last QK^T is done
                    if (j == 0) load_q();
                }
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer (leader)
        if (rank == 0 && lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(256, 128, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(256, 128, true);
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
                const uint64_t da = desc_base(sb + kQOff + t * kQTile, 16);
                const uint64_t db = desc_base(sb + kKOff + ks * kKTile, 16);
#pragma unroll
                for (int s = 0; s < DQK / 16; ++s)
                    mma_ss_pair(tmem + col_s(t), da + (uint64_t)(((s >> 2) * kQBox + (s & 3) * 32) >> 4),
                                db + (uint64_t)(((s >> 2) * kKBox + (s & 3) * 32) >> 4), idesc_qk, s > 0 ? 1u : 0u);
            };
            auto issue_pv = [&](int t, int vs, bool acc) {
                const uint64_t dv = desc_base(sb + kVOff + vs * kVTile, kQBox);
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_ts_pair(tmem + col_o(t), tmem + col_s(t) + 8 * s, dv + (uint64_t)(s * 2048 >> 4), idesc_pv,
                                (acc || s > 0) ? 1u : 0u);
            };
            int kc = 0;
            for (int k = 0, w = item_index(0); w < p.n_work; ++k, w = item_index(k)) {
                const Item it = make_item(p, w);
                const int n = it.n_kt;
                pair_wait(bar(kBarKReady + kc % kKStages), (kc / kKStages) & 1, p.wait, abort);
                for (int t = 0; t < 2; ++t) {
                    pair_wait(bar(kBarQReady + t), k & 1, p.wait, abort);
                    tc_fence_after();
                    issue_qk(t, kc % kKStages);
                    commit_pair(bar(kBarSFull + t));
                    if (n == 1) commit_pair(bar(kBarQEmpty + t));
                }
                for (int j = 0; j < n; ++j) {
                    const int g = kc + j;
                    const bool nxt = j + 1 < n;
                    const bool last_qk = j + 2 == n;
                    const int ks = (g + 1) % kKStages, vs = g % kVStages;
                    pair_wait(bar(kBarPReady + 0), g & 1, p.wait, abort);
                    tc_fence_after();
                    issue_pv(0, vs, j > 0);
                    if (nxt) {
                        pair_wait(bar(kBarKReady + ks), ((g + 1) / kKStages) & 1, p.wait, abort);
                        tc_fence_after();
                        issue_qk(0, ks);
                        commit_pair(bar(kBarSFull + 0));
                        if (last_qk) commit_pair(bar(kBarQEmpty + 0));
                    } else {
                        commit_pair(bar(kBarODone + 0));
                    }
                    pair_wait(bar(kBarPReady + 1), g & 1, p.wait, abort);
                    tc_fence_after();
                    issue_pv(1, vs, j > 0);
                    commit_pair(bar(kBarVEmpty + vs));
                    if (nxt) {
                        issue_qk(1, ks);
                        commit_pair(bar(kBarSFull + 1));
                        if (last_qk) commit_pair(bar(kBarQEmpty + 1));
                    } else {
                        commit_pair(bar(kBarODone + 1));
                    }
                }
                kc += n;
            }
        }
    } else if (warp >= kWarpRope && warp < kWarpTma) {
        // ------------------------------------------------------------ K RoPE (both CTAs, 64 keys each)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsRope));
        const int rt = threadIdx.x - kWarpRope * 32;
        const int c = rt & 7, r0 = rt >> 3;
        const int max_row = p.rope.max_pos - 1;
        const int half0 = 64 * (int)rank;
        KHalfRope<C::kRopeBoxes, C::kRopeBox0> kr;
        if (KROT) kr.init(p.rope.cs, c);
        int kc = 0;
        for (int k = 0, w = item_index(0); w < p.n_work; ++k, w = item_index(k)) {
            const Item it = make_item(p, w);
            if (q_shared(KROT, p.G)) {
                // this CTA's share of the item's Q tiles: heads [hs, G) of both
                const int hs = q_heads_softmax(p.G);
                for (int t = 0; t < 2; ++t) {
                    const int T = 2 * (int)rank + t;
                    pair_wait(bar(kBarQFull + t), k & 1, p.wait, abort);
                    const bool mine = p.G < 16 || (rt >> 6) == t;  // G = 16: threads 64 t .. 64 t + 63
                    if (mine)
                        rope_q_part<C::kRopeBoxes, C::kRopeBox0>(
                            smem + kQOff + t * kQTile, p.rope.cs, p.q_pos0 + it.r0 + T * P, P,
                            min(P, p.S_q - (it.r0 + T * P)), p.G < 16 ? rt : (rt & 63), p.G < 16 ? 128 : 64, hs, p.G);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) arrive_leader(bar(kBarQReady + t));
                }
            }
            if (KROT) kr.load_seed(p.rope.cs, min(128 * it.j_lo + half0 + r0, max_row), c);
            for (int j = 0; j < it.n_kt; ++j, ++kc) {
                const int ks = kc % kKStages;
                pair_wait(bar(kBarKFull + ks), (kc / kKStages) & 1, p.wait, abort);
                if (KROT && !p.keys_prerotated) kr.rotate(smem + kKOff + ks * kKTile, rt);
                if (KROT && j + 1 < it.n_kt)
                    kr.load_seed(p.rope.cs, min(128 * (it.j_lo + j + 1) + half0 + r0, max_row), c);
                // K(j) ready also means V(j) has landed: the MMA thread waits for
                // KReady(j) before QK(j), which precedes PV(j)
                pair_wait(bar(kBarVFull + kc % kVStages), (kc / kVStages) & 1, p.wait, abort);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) arrive_leader(bar(kBarKReady + ks));
            }
        }
    } else if (warp < kWarpRope) {
        // ------------------------------------------------------------ softmax + epilogue (both CTAs)
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        const int t = warp >> 2;
        const int T = 2 * (int)rank + t;       // tile of the item
        const int i = (warp & 3) * 32 + lane;  // row of the M tile == TMEM lane
        const int W = p.window;
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t s_addr = lane_base + col_s(t);
        const uint32_t o_addr = lane_base + col_o(t);
        auto rotate_q = [&](const Item &it, int k) {
            pair_wait(bar(kBarQFull + t), k & 1, p.wait, abort);
            if (q_shared(KROT, p.G)) {
                const int hs = q_heads_softmax(p.G);
                if (p.G < 16)
                    rope_q_part<C::kRopeBoxes, C::kRopeBox0>(smem + kQOff + t * kQTile, p.rope.cs,
                                                             p.q_pos0 + it.r0 + T * P, P,
                                                             min(P, p.S_q - (it.r0 + T * P)), i, 128, 0, hs);
                else  // G = 16: two threads per combo, 6 heads each
                    rope_q_part<C::kRopeBoxes, C::kRopeBox0>(smem + kQOff + t * kQTile, p.rope.cs,
                                                             p.q_pos0 + it.r0 + T * P, P,
                                                             min(P, p.S_q - (it.r0 + T * P)), i >> 1, 128,
                                                             6 * (i & 1), 6 * (i & 1) + 6);
            } else {
                rope_q_tile<C::kRopeBoxes, C::kRopeBox0>(smem + kQOff + t * kQTile, i, p.rope.cs,
                                                         p.q_pos0 + it.r0 + T * P, p.G, P,
                                                         min(P, p.S_q - (it.r0 + T * P)));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) arrive_leader(bar(kBarQReady + t));
        };
        int kc = 0;
        if (item_index(0) < p.n_work) rotate_q(make_item(p, item_index(0)), 0);
        for (int k = 0, w = item_index(0); w < p.n_work; ++k, w = item_index(k)) {
            const Item it = make_item(p, w);
            const int r = it.r0 + T * P + i % P;  // query row index
            const int m = p.q_pos0 + r;           // its position
            const bool in_prefix = m < p.prefix_len;
            const int key_lo = (in_prefix || W <= 0) ? 0 : m - W + 1;
            const int key_hi = in_prefix ? p.prefix_len - 1 : m;
            float m_run = -INFINITY, l_run = 0.f;

            for (int j = 0; j < it.n_kt; ++j) {
                pair_wait(bar(kBarSFull + t), (kc + j) & 1, p.wait, abort);
                tc_fence_after();
                const int kstart = 128 * (it.j_lo + j);
                const int hi_c = key_hi - kstart;
                const int lo_c = key_lo - kstart;
                const bool full_vis = lo_c <= 0 && hi_c >= 127;
                const bool all_full = __all_sync(0xffffffffu, full_vis);
                uint32_t v[128];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    tmem_ld32(s_addr + 32 * ch, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * ch]));
                tmem_wait_ld();
                if (!all_full) mask_row128(v, lo_c, hi_c);
                float acc[8];
#pragma unroll
                for (int a = 0; a < 8; ++a) acc[a] = __uint_as_float(v[a]);
#pragma unroll
                for (int e = 8; e + 16 <= 128; e += 16)
#pragma unroll
                    for (int a = 0; a < 8; ++a)
                        acc[a] = fmax3(acc[a], __uint_as_float(v[e + a]), __uint_as_float(v[e + 8 + a]));
#pragma unroll
                for (int a = 0; a < 8; ++a) acc[a] = fmaxf(acc[a], __uint_as_float(v[120 + a]));
                const float mx =
                    fmax3(fmax3(acc[0], acc[1], acc[2]), fmax3(acc[3], acc[4], acc[5]), fmaxf(acc[6], acc[7]));
                const float m_tile = mx * p.scale_log2;
                const float m_new = fmaxf(m_run, m_tile);
                const bool need = (m_run != -INFINITY) && (m_new > m_run + 8.f);
                if (__any_sync(0xffffffffu, need)) {
                    const float alpha = (m_new == -INFINITY) ? 1.f : fast_exp2(m_run - m_new);
                    l_run *= alpha;
                    m_run = m_new;
#pragma unroll 1
                    for (int ch = 0; ch < DV / 16; ++ch) {
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
                const uint64_t SC = f2_pack(p.scale_log2, p.scale_log2);
                const uint64_t NM = f2_pack(-m_use, -m_use);
                uint64_t lacc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e2 = 0; e2 < 16; ++e2) {
                        const uint64_t x =
                            f2_pack(__uint_as_float(v[32 * q4 + 2 * e2]), __uint_as_float(v[32 * q4 + 2 * e2 + 1]));
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
                if (lane == 0) arrive_leader(bar(kBarPReady + t));
            }
            kc += it.n_kt;

            const int w_next = item_index(k + 1);
            if (w_next < p.n_work) rotate_q(make_item(p, w_next), k + 1);

            // ---- epilogue: O / l -> bf16 -> global, one row per thread
            pair_wait(bar(kBarODone + t), k & 1, p.wait, abort);
            tc_fence_after();
            const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
            if constexpr (C::kTmaStoreO) {
                // The warp's 32 rows go to its staging buffer as two swizzled
                // [32 rows][64 dims] boxes (box row == lane: rows are head-major,
                // P positions per head), then leave by two TMA stores; rows past
                // S_q fall outside the tensor and are not written.
                uint8_t *stage = smem + C::kStageOff + warp * C::kStageWarpBytes;
                if (lane == 0) bulk_wait_group_read0();  // the previous item's stores have read it
                __syncwarp();
#pragma unroll
                for (int ch = 0; ch < DV / 32; ++ch) {
                    uint32_t o[32];
                    tmem_ld32(o_addr + 32 * ch, o);
                    tmem_wait_ld();
                    uint32_t w2[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        w2[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
                    uint8_t *half = stage + (ch >> 1) * (C::kStageWarpBytes / 2);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        *reinterpret_cast<uint4 *>(half + swz128(lane, (ch & 1) * 4 + q4)) =
                            make_uint4(w2[4 * q4], w2[4 * q4 + 1], w2[4 * q4 + 2], w2[4 * q4 + 3]);
                }
                tc_fence_before();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int wq = 32 * (warp & 3);          // the warp's first M-tile row
                    const int y = it.r0 + T * P + wq % P;    // its output row (query index)
                    if (y < p.S_q) {
                        tma_store_4d(&tm_o, smem_u32(stage), 0, y, wq / P, it.unit);
                        tma_store_4d(&tm_o, smem_u32(stage) + C::kStageWarpBytes / 2, 64, y, wq / P, it.unit);
                    }
                    bulk_commit_group();
                }
            } else {
                const int hl = i / P;
                uint4 *dst = reinterpret_cast<uint4 *>(p.out + ((size_t)(it.zq + hl) * p.S_q + r) * DV);
#pragma unroll
                for (int ch = 0; ch < DV / 32; ++ch) {
                    uint32_t o[32];
                    tmem_ld32(o_addr + 32 * ch, o);
                    tmem_wait_ld();
                    uint32_t w2[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        w2[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
                    if (r < p.S_q) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            dst[4 * ch + q4] =
                                make_uint4(w2[4 * q4], w2[4 * q4 + 1], w2[4 * q4 + 2], w2[4 * q4 + 3]);
                    }
                }
                tc_fence_before();
            }
        }
        // the last item's stores have completed before the CTA (and its shared memory) goes
        if (C::kTmaStoreO && lane == 0) bulk_wait_group0();
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync();  // every MMA of the pair has completed and every remote arrival has landed
    if (warp == kWarpMma) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
    }
}

template <int DQK, int DR, bool KROT>
cudaError_t launch_pair_t(const PrefillLaunch &L, cudaStream_t stream)
{
    using C = PairCfg<DQK, DR>;
    cudaError_t err = cudaFuncSetAttribute(prefill_pair_kernel<DQK, DR, KROT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           C::kSmemBytes);
    if (err != cudaSuccess) return err;
    // setmaxnreg.inc blocks until the block's own pool can serve it: never
    // launch unless the split fits the registers the block is launched with
    cudaFuncAttributes fa;
    err = cudaFuncGetAttributes(&fa, prefill_pair_kernel<DQK, DR, KROT>);
    if (err != cudaSuccess) return err;
    if (fa.numRegs < kLaunchRegs) return cudaErrorInvalidConfiguration;
    return launch_dependent(prefill_pair_kernel<DQK, DR, KROT>, L.grid, kThreads, C::kSmemBytes, stream, L.tm_q, L.tm_k,
                            L.tm_v, L.tm_o, L.p);
}

}  // namespace

cudaError_t launch_prefill_pair(const PrefillLaunch &L, cudaStream_t stream)
{
    if (L.grid & 1) return cudaErrorInvalidValue;
    if (L.p.d_h == 128 && L.p.d_rope == 128)
        return L.p.keys_prerotated ? launch_pair_t<128, 128, false>(L, stream) : launch_pair_t<128, 128, true>(L, stream);
    if (L.p.d_h == 192 && L.p.d_rope == 64)
        return L.p.keys_prerotated ? launch_pair_t<192, 64, false>(L, stream) : launch_pair_t<192, 64, true>(L, stream);
    return cudaErrorInvalidValue;
}

}  // namespace apex
