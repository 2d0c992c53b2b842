// decode.cuh - one KV-cache decode step (declarations).
#pragma once

#include "common.cuh"

namespace smol {

struct DecodeArgs {
  smol_config cfg;
  int B, S_max;
  const int *ids;          // [B]
  const int *cache_len;    // [B]
  const bf16 *k_cache, *v_cache;   // [L, B, KV, S_max, hd]
  bf16 *k_new, *v_new;     // [L, B, KV, hd]
  bf16 *logits;            // [B, V]
  const float2 *rope;      // two-level (cos, sin) table, see rope_table_rows
  const bf16 *embed;       // bf16 table for the gather
  const f16 *head;         // f16 norm-folded tied head
  const uint8_t *layer0;   // first packed layer
  size_t layer_bytes, off_qkv, off_o, off_gu, off_down;
  int *next;               // [B] or nullptr: the greedy next token of each row (first maximum
                           // of the bf16 logits), taken in the head GEMM's epilogue; logits
                           // may then be nullptr
};

size_t decode_ws_bytes(const smol_config *cfg, int B);
cudaError_t run_decode(const DecodeArgs &a, void *ws, int sms, cudaStream_t stream, int *launches);

}  // namespace smol
