// Internal layout of the pinned host KV pool (opaque to ABI users).
#pragma once

#include <stdint.h>

#include <vector>

struct ig_pool {
  int layers = 0, B = 0, H = 0, d = 0, cap = 0;
  int policy = 0;            // IG_POOL_COUNTER, IG_POOL_FIFO or IG_POOL_LRU
  bool storage = true;       // false: the slot manager only, no K/V rows
  int qbits = 0;             // 0: fp16 rows; 8: e4m3 codes, 4: int4 codes, one fp32 scale per row
  uint8_t* R = nullptr;      // quantized pools: pinned, mapped code records [layers][B][H][cap][rec]:
  int rec = 0;               //   K codes, then V codes (d * qbits / 8 bytes each; rec = 128 or 256
                             //   bytes at d = 128, whole 128-byte lines)
  float* S = nullptr;        // quantized pools: the rows' fp32 scales in device memory
                             //   [layers][B][H][cap][2] (K, V)
  int sdev = -1;             // the device that holds S
  uint16_t* K = nullptr;     // pinned, mapped host memory [layers][B][H][cap][d]
  uint16_t* V = nullptr;
  uint16_t* Kdev = nullptr;  // the same memory as seen from the device
  uint16_t* Vdev = nullptr;
  std::vector<uint8_t> counter;   // [layers][B][cap]
  std::vector<uint32_t> seq;      // insertion order per slot, [layers][B][cap]
  std::vector<int32_t> filled;    // resident slots, [layers][B]
  std::vector<uint32_t> next_seq; // [layers][B]
  std::vector<uint32_t> last_use; // LRU time of each slot, [layers][B][cap]
  std::vector<uint32_t> clock;    // LRU time (updates folded so far), [layers][B]
  std::vector<int64_t> evictions; // placements into a full pool, [layers][B]
};
