// decode_tag.h -- the tags of the fused decode kernel's hand-off words, in host and device
// code alike (the arithmetic is also checked on the CPU).
//
// Every value one CTA hands to another in the decode kernel travels as a 64-bit word
// {32-bit payload, 32-bit tag}.  The tag names the launch and the layer: (epoch + 1) * 64
// + layer, where the epoch counts the launches that used the same tables, modulo
// DEC_EPOCH_PERIOD.  Within one period every (epoch, layer) pair has its own tag, no tag
// is 0 (the value of a word that was never written) and no tag overflows 32 bits.  When
// the epoch wraps back to 0, the launch that ends the period clears every tagged word, so
// no word written in the old period can carry a tag of the new one.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define MOE_HD __host__ __device__
#else
#define MOE_HD
#endif

namespace moe {

constexpr int DEC_TAG_LAYER_BITS = 6;                        // up to 64 layers per launch
constexpr uint32_t DEC_EPOCH_PERIOD = (1u << (32 - DEC_TAG_LAYER_BITS)) - 1u;

MOE_HD constexpr uint32_t dec_tag(uint32_t epoch, int layer) {
  return ((epoch + 1u) << DEC_TAG_LAYER_BITS) + static_cast<uint32_t>(layer);
}

// The epoch of the next launch; 0 after the last epoch of a period.
MOE_HD constexpr uint32_t dec_next_epoch(uint32_t epoch) { return epoch + 1u >= DEC_EPOCH_PERIOD ? 0u : epoch + 1u; }

}  // namespace moe
