// Parameters shared by the host launcher and the split / merge kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

struct SplitParams {
  // query / outputs
  const uint16_t* q;        // bf16 [T, Hq, D], head stride D
  int64_t q_stride_t;       // elements
  uint16_t* out;            // bf16 [T, Hq, D]
  int64_t out_stride_t, out_stride_h;
  float* lse;               // f32 [T, Hq] or nullptr
  int64_t lse_stride_t, lse_stride_h;
  // paged metadata
  const int32_t* block_tables;
  int64_t bt_stride;
  const int32_t* seq_lens;
  const int32_t* qsl;       // [B+1] or nullptr (one token per sequence)
  int32_t num_seqs;         // B
  int32_t num_tokens;       // T (rows of q / out)
  int32_t Hq, Hkv, G;
  int32_t max_qlen;
  int32_t num_pages;        // NB
  int32_t max_blocks;       // block-table columns
  // plan
  int32_t HC;               // KV heads per CTA
  int32_t NC;               // head chunks = Hkv / HC
  int32_t MT;               // 16-row tiles per head
  int32_t R_max;            // G * max_qlen rows per head
  int32_t nstage;
  int32_t min_pages;        // minimum pages of work per CTA
  int32_t pair_pages;       // consumers take two pages of a segment at once
  int32_t window;           // sliding window (keys p-W < j <= p), 0 = off
  const float* sinks;       // [Hq] sink logits or nullptr
  // math
  float scale_log2;         // scale * k_scale * log2(e)
  float v_scale;            // applied to the output (1 for bf16 caches)
  // workspace
  int4* ws_unit;            // [B * NC] per unit: {first CTA, pieces | first-is-tail << 30, t0, qn}
  float2* ws_ml;            // [2 * grid][HC][R_max] (running max in log2 units, sum)
  float* ws_o;              // [2 * grid][HC][R_max][D] unnormalised partial outputs
  uint32_t* err;            // device status word
  // shared-memory layout (bytes from the 1024-aligned base)
  uint32_t off_prefix;      // int32 [B+1] page prefix, then [B] seq_lens, then [B+1] query starts
  uint32_t off_bar;
  uint32_t off_q;
  uint32_t q_slot_bytes;
  uint32_t off_stage;
  uint32_t stage_bytes;     // K tiles + V tiles of one page
  uint32_t kv_bytes;        // K (or V) tiles of one page: HC * 16 * D * elem
  int32_t block_pages;      // tensor-memory variant: pages per ring stage (block)
  uint32_t off_xchg;        // tensor-memory variant: softmax warps' exchange buffers (4 KB)
  // per-token fp8 scales (token-scale variant of the split kernel): f32 [NB, Hkv, 16],
  // staged per page behind the K and V tiles: [HC][16] K scales, then [HC][16] V scales
  const float* k_tok;
  const float* v_tok;
  int64_t tok_stride_page;  // floats between pages of the scale tensors
  uint32_t tok_bytes;       // HC * 16 * 4: one tensor's scales of one page
  // MLA kernel: bytes between the shared-memory regions of a CTA's teams,
  // query slots per team (1 or 2); tensor-memory MLA kernel: slots of the Q
  // staging ring
  uint32_t team_bytes;
  int32_t q_slots;
  // tensor-memory MLA kernel: the three block buffers (rows in the MMA layout)
  uint32_t off_buf;
  // pipeline waits give up after wait_ns nanoseconds (status bit 3)
  uint64_t wait_ns;
  // testing aid (mma.sync kernel): the producer of split CTA starve_cta issues
  // no copies, so that CTA's consumers run into the wait limit; -1 = none
  int32_t starve_cta;
  // tensor-memory MLA kernel: the Q staging ring; pages the work split
  // charges for every unit a CTA starts (0: an equal page split)
  uint32_t off_qring;
  int32_t seg_cost;
};

struct MergeParams {
  uint16_t* out;
  int64_t out_stride_t, out_stride_h;
  float* lse;
  int64_t lse_stride_t, lse_stride_h;
  const int32_t* seq_lens;
  const int32_t* qsl;
  int32_t num_seqs, num_tokens;
  int32_t G, HC, NC, R_max, max_qlen;
  int32_t split_grid;       // CTAs the split kernel was launched with
  float v_scale;
  const int4* ws_unit;
  const float2* ws_ml;
  const float* ws_o;
  uint32_t* err;
};

struct CacheWriteParams {
  const uint16_t* key;      // bf16 [T, Hkv, D]
  const uint16_t* value;
  int64_t k_stride_t, k_stride_h, v_stride_t, v_stride_h;   // elements
  const int32_t* slot_mapping;   // [T]
  uint8_t* k_cache;         // [NB, 16, Hkv, D] bf16 or e4m3 bytes
  uint8_t* v_cache;
  int64_t kc_stride_page, kc_stride_slot, kc_stride_head;   // elements of the cache dtype
  int64_t vc_stride_page, vc_stride_slot, vc_stride_head;
  int32_t num_tokens, num_kv_heads, head_dim, num_pages;
  float k_scale, v_scale;   // fp8 only: code = e4m3(x / scale), one IEEE fp32 division
  uint32_t* err;
  // per-token quantisation (fp8 only): row scale = amax / 448 stored at
  // [page, head, slot] of f32 [NB, Hkv, 16] tensors; nullptr = per-tensor scales
  float* k_tok;
  float* v_tok;
  int64_t ks_stride_page, ks_stride_head, ks_stride_slot;   // floats
  int64_t vs_stride_page, vs_stride_head, vs_stride_slot;
};

// Grid sized to one wave of resident blocks on num_sms SMs (occupancy taken
// once by init_cache_write_occupancy, outside any stream capture).
cudaError_t launch_cache_write(bool fp8, const CacheWriteParams& p, int num_sms, cudaStream_t stream);
void init_cache_write_occupancy();

// Launchers (one translation unit per cache dtype).  `pdl` requests
// programmatic dependent launch for the merge kernel.
cudaError_t launch_split_bf16(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                              int grid, int threads, int smem, bool pdl, cudaStream_t stream);
cudaError_t launch_split_fp8(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                             int grid, int threads, int smem, bool pdl, cudaStream_t stream);
// fp8 caches with per-token scales (p.k_tok / p.v_tok set).
cudaError_t launch_split_fp8_tok(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                                 int grid, int threads, int smem, bool pdl, cudaStream_t stream);
cudaError_t set_split_smem_limits_fp8_tok(int smem);
// wide: one 256-thread block per (unit, row), threads across partials (many
// partials per unit); otherwise one warp per (unit, row), 8 rows per block.
cudaError_t launch_merge(int head_dim, const MergeParams& p, int units, int rows, bool wide, bool pdl,
                         cudaStream_t stream);
// Tensor-memory (tcgen05) variant for up to 128 query rows per KV head (bf16
// caches, one KV head per CTA, 192 threads).
cudaError_t launch_split_tc(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& p,
                            int grid, int smem, bool pdl, cudaStream_t stream);
cudaError_t set_split_smem_limits_tc(int smem);
// MLA decode over a latent cache [NB, 16, 576] (value = first 512 columns);
// rt = 16-row tiles of a head chunk (1 or 2).  A CTA runs mla_teams(rt)
// independent teams in mla_threads(rt) threads; p.HC = 1, p.G = heads per chunk.
cudaError_t launch_mla(bool fp8, int rt, const CUtensorMap& tm, const SplitParams& p, int grid, int smem, bool pdl,
                       cudaStream_t stream);
int mla_threads(int rt);
int mla_teams(int rt);
cudaError_t set_mla_smem_limits(int smem);
// Tensor-memory (tcgen05) MLA decode: one head chunk of at most rpad (16 or
// 32) query rows per unit, mla_tc_threads() threads a CTA; shared-memory
// layout in p.off_buf (block buffers), p.off_q (P buffers), p.off_stage (fp8:
// raw page ring of p.nstage slots), p.off_bar, p.off_xchg, p.off_prefix.  tm:
// a whole page per box (fp8), tb: one 64-feature column block of a page per
// box (bf16).
cudaError_t launch_mla_tc(bool fp8, int rpad, const CUtensorMap& tm, const CUtensorMap& tb, const SplitParams& p,
                          int grid, int smem, bool pdl, cudaStream_t stream);
int mla_tc_threads();
cudaError_t set_mla_tc_smem_limits(int smem);
// LSE merge of MLA partials (512 value columns; the split kernel writes each
// piece's normalised output in f16 into ws_o): one warp per (unit, row).
cudaError_t launch_merge_mla(const MergeParams& p, int units, int rows, bool pdl, cudaStream_t stream);
cudaError_t set_split_smem_limits_bf16(int smem);
// Resolve the no-allocation entry point's static scratch on the current device
// (once per device; part of the per-device set-up).  Returns a pa_status.
int static_scratch_setup();
cudaError_t set_split_smem_limits_fp8(int smem);

}  // namespace pa
