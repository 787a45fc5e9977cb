// kernel_params.h -- plain parameter blocks passed from the host library to
// the kernels, and the launch entry points each kernel file provides.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace apex {

// Codes a kernel may leave in the per-device status word.
constexpr uint32_t kStatusWaitTimeout = 1;

struct WaitCtl {
    uint32_t *status;     // per-device status word (device memory)
    uint64_t timeout_ns;  // bound on any single wait
};

// Bound on a single kernel wait: APEX_ATTN_WAIT_TIMEOUT_MS milliseconds when
// that variable holds a positive number, else 2 s (read once per process).
uint64_t wait_timeout_ns();

// (cos, sin)(pos * theta_i) for pos in [0, max_pos), i in [0, d_h/2), fp32,
// row-major [max_pos][d_h/2].
struct RopeTableView {
    const float2 *cs;
    int max_pos;
};

// ----------------------------------------------------------------- decode
constexpr int kDecodeKeysPerStage = 64;  // keys per pipeline stage
constexpr int kDecodeMaxSplit = 4096;    // hard cap on KV splits per (b, kv-head)

struct DecodeParams {
    const uint16_t *q;  // [B, H_q, 1, d_h] bf16
    uint16_t *out;      // [B, H_q, 1, d_h] bf16
    float *ws_o;        // [B*H_q, n_split, d_h]  partial outputs (unnormalised)
    float2 *ws_ml;      // [B*H_q, n_split]       partial (max (log2 units), sum)
    RopeTableView rope;
    WaitCtl wait;
    int B, H_q, H_kv, G, S_k, d_h;
    int q_pos;              // query position
    int k_lo;               // first visible key
    int k_hi;               // last visible key (q_pos, or P - 1 for a query inside a prefix of P)
    int stage0;             // first stage index (stage s covers keys [64 s, 64 s + 64))
    int n_stages;           // stages per (b, kv-head)
    int n_split;            // splits per (b, kv-head)
    int stages_per_split;   // last split may have fewer
    int n_items;            // B * H_kv * n_split
    float scale_log2;       // log2(e) / sqrt(d_h)
    int d_v;                // value / output row length (d_h for the plain block)
    int d_rope;             // trailing q / k entries RoPE turns (d_h for the plain block)
};

struct DecodeLaunch {
    CUtensorMap tm_k, tm_v;  // 3-D maps over [B*H_kv, S_k, d_h], box {64, 64, 1}, 128B swizzle
    DecodeParams p;
    int grid;                // CTAs of the split kernel (persistent)
};

// keys_prerotated selects the variant that uses the cached keys as they are
cudaError_t launch_decode(const DecodeLaunch &L, bool keys_prerotated, cudaStream_t stream);
int decode_ctas_per_sm(int d_qk, int d_v, int G);

// ----------------------------------------------------------------- prefill
struct PrefillParams {
    uint16_t *out;  // [B, H_q, S_q, d_h] bf16
    RopeTableView rope;
    WaitCtl wait;
    int B, H_q, H_kv, G, S_q, S_k, d_h;
    int window;     // <= 0: none
    int q_pos0;
    int prefix_len;       // bidirectional prefix [0, P); 0: none
    int keys_prerotated;  // keys already rotated: no K RoPE
    int rows_per_head;   // query positions per head in one 128-row M tile (128 / G)
    int n_qblocks;       // position blocks per (b, kv-head); a block = 2 M tiles (4 on CTA pairs)
    int n_work;          // B * H_kv * n_qblocks (work items, walked by a persistent grid)
    float scale_log2;    // log2(e) / sqrt(d_h)
    int d_rope;          // trailing entries of a q / k row that RoPE turns (d_h: all)
};

struct PrefillLaunch {
    CUtensorMap tm_q, tm_k, tm_v;
    // CTA-pair kernel: 4-D map over out viewed as [B*H_kv][G][S_q][128] (the G
    // query heads of a KV head adjacent), box {64, min(P, 32), max(1, 32 / P), 1}
    // with P = 128 / G: one box is the 64-dim half of the 32 M-tile rows of one
    // warp; 128-byte swizzle; elements outside the tensor are not written
    CUtensorMap tm_o;
    PrefillParams p;
    int grid;  // persistent CTAs (at most one per SM)
};

cudaError_t launch_prefill(const PrefillLaunch &L, cudaStream_t stream);
// CTA-pair variant: tm_k's box is {64, 64, 1}, grid even, blocks of 4 M tiles; value and
// output rows of 128; (d_h, d_rope) = (128, 128) for the plain block or (192, 64) for
// decoupled RoPE (d_h is then the q / k row length)
cudaError_t launch_prefill_pair(const PrefillLaunch &L, cudaStream_t stream);

// ----------------------------------------------------------------- key rotation
struct RopeKeysParams {
    const uint16_t *in;
    uint16_t *out;
    long long in_stride, out_stride;  // elements between heads
    int n_heads, n_pos, pos0;
    int d_row;  // entries per key row
    int d_rot;  // trailing entries of a row that are rotated (the rest are copied)
    RopeTableView rope;
};

cudaError_t launch_rope_keys(const RopeKeysParams &p, int sm_count, cudaStream_t stream);

// ----------------------------------------------------------------- self-test
// one CTA whose bounded mbarrier wait can never complete (reports kStatusWaitTimeout)
cudaError_t launch_wait_selftest(const WaitCtl &wc, cudaStream_t stream);

}  // namespace apex
