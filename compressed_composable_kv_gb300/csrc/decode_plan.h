// Work decomposition of one decode step (one layer, a batch of sequences):
// the key tiles of every (sequence, kv head) unit, laid end to end, are cut
// into equal contiguous ranges, one per CTA of the launch, so every SM
// streams the same number of tiles whatever the sequences' lengths.  A CTA's
// range may start or end inside a unit; the CTAs sharing a unit each write a
// partial result (m, l, O) and the last one to finish merges them.
//
// Everything here is computed from the device-side lengths inside the kernel
// (so a captured launch replays with new lengths), and is also compiled for
// the host so the decomposition can be checked on the CPU.
#pragma once

#include <stdint.h>

namespace c2kv {

constexpr int kDecKeyTile = 128;       // keys per tile
constexpr int kDecMaxSeqs = 16;        // sequences per launch
constexpr int kDecMaxCtas = 256;       // CTAs per launch (one per SM)
constexpr int kDecClusterTilesPerSm = 8;   // below this many tiles per SM, prefer the cluster merge

struct DecodeMap {
  int32_t nseq, hkv, ctas;
  int32_t tb[kDecMaxSeqs];             // tiles of each unit of sequence b (0: sequence skipped)
  int64_t start[kDecMaxSeqs + 1];      // global index of sequence b's first tile
  int64_t total;                       // tiles of the launch
};

// keys[b]: keys sequence b attends over (cached + the new one); a value < 1
// marks a sequence to skip.  Unit (b, h) holds global tiles
// [start[b] + h * tb[b], start[b] + (h + 1) * tb[b]).
__host__ __device__ inline void decode_map_build(DecodeMap& m, const int32_t* keys, int nseq, int hkv, int ctas) {
  m.nseq = nseq;
  m.hkv = hkv;
  m.ctas = ctas;
  int64_t acc = 0;
  for (int b = 0; b < kDecMaxSeqs; ++b) {
    const int32_t kb = b < nseq ? keys[b] : 0;
    m.start[b] = acc;
    m.tb[b] = kb > 0 ? (kb + kDecKeyTile - 1) / kDecKeyTile : 0;
    acc += (int64_t)m.tb[b] * hkv;
  }
  m.start[kDecMaxSeqs] = acc;
  m.total = acc;
}

// CTA c owns global tiles [decode_cta_first(c), decode_cta_first(c + 1)).
__host__ __device__ inline int64_t decode_cta_first(const DecodeMap& m, int c) {
  return m.total == 0 ? 0 : (int64_t)c * m.total / m.ctas;
}

// The CTA whose range holds global tile x (0 <= x < total): the c with
// floor(c T / C) <= x < floor((c + 1) T / C), i.e. c = ceil((x + 1) C / T) - 1.
__host__ __device__ inline int decode_cta_of(const DecodeMap& m, int64_t x) {
  return (int)(((x + 1) * m.ctas - 1) / m.total);
}

struct DecodeTile {
  int32_t b, h, t;   // sequence, kv head, tile within the unit
};

// Global tile x (0 <= x < total) as (sequence, kv head, tile of the unit).
__host__ __device__ inline DecodeTile decode_locate(const DecodeMap& m, int64_t x) {
  int b = 0;
  while (b + 1 < kDecMaxSeqs && x >= m.start[b + 1]) ++b;
  const int64_t r = x - m.start[b];
  DecodeTile d;
  d.b = b;
  d.h = (int)(r / m.tb[b]);
  d.t = (int)(r % m.tb[b]);
  return d;
}

// The tile after `d` in global order (valid while the result is < total).
__host__ __device__ inline DecodeTile decode_next(const DecodeMap& m, DecodeTile d) {
  if (++d.t < m.tb[d.b]) return d;
  d.t = 0;
  if (++d.h < m.hkv) return d;
  d.h = 0;
  do {
    ++d.b;
  } while (d.b < kDecMaxSeqs && m.tb[d.b] == 0);
  return d;
}

// With fewer tiles than CTAs some CTAs own no tile.
__host__ __device__ inline bool decode_cta_empty(const DecodeMap& m, int c) {
  return decode_cta_first(m, c) == decode_cta_first(m, c + 1);
}

// Partial-result slots: CTA c writes slot 2c for its first segment and slot
// 2c + 1 for its last one (when they differ); a segment covering its whole
// unit writes the output directly and takes no slot.  The CTAs sharing unit
// (b, h) are the non-empty ones in [cta_of(first tile), cta_of(last tile)];
// the slot such a CTA c wrote for the unit is:
__host__ __device__ inline int decode_slot_of(const DecodeMap& m, int c, int64_t unit_first) {
  return 2 * c + (decode_cta_first(m, c) < unit_first ? 1 : 0);
}

}  // namespace c2kv
