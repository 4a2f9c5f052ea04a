// lamp_qkv.cuh -- parameters of the QKV projection kernel (lamp_qkv.cu).
#pragma once
#include <cstdint>
#include <cuda.h>

namespace lamp {

// QKV projection parameters (see lamp_qkv.cu).
struct QkvParams {
  CUtensorMap tmX, tmW;          // x [T, hidden], W [ncols, hidden]: BF16, K-major
  uint16_t* q;                   // [B, N, Hq, D]  BF16
  uint16_t* k;                   // [B, N, Hkv, D] BF16
  uint16_t* v;                   // [B, N, Hkv, D] BF16
  uint8_t* k8;                   // workspace [B, Hkv, N, D] E4M3
  uint16_t* v16;                 // workspace [B, Hkv, N, D] fp16
  uint8_t* q8;                   // workspace [B, Hq, N, D] E4M3
  float* nq;                     // workspace [B, Hq, N]: norm of each E4M3 query row
  float* nqc;                    // workspace [B, Hq, N, D/32]: norms of its 32-element chunks
  float* nk;                     // workspace [B, Hkv, T_k] (zeroed before the launch)
  float* nkc;                    // workspace [B, Hkv, T_k, D/32] (zeroed before the launch)
  unsigned int* abort;           // grid abort word (zeroed before the launch)
  unsigned long long* counters;  // optional: status slot 9 on a timed-out wait
  unsigned long long timeout_ns;
  int B, N, Hq, Hkv, D, T, hidden, ncols;  // T = B N tokens, ncols = (Hq + 2 Hkv) D
};

}  // namespace lamp
