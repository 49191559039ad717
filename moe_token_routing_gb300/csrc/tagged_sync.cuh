// Hand-off of 32-bit values between the CTAs of one grid through 64-bit words
// that carry a per-call tag in their upper half.
//
// A producer stores {tag, value} with one 64-bit store; a consumer checks that
// the word carries the current call's tag. The value arrives together with
// the tag in one single-copy-atomic access, so no fence is needed: a stale
// word from an earlier call carries an older tag and is simply not ready yet.
// To keep many consumers from polling many words, producers also bump a
// relaxed counter once their words are stored; consumers poll that one word
// first and then check the tags (waiting on any word that is still behind).
// Every wait is bounded (kSyncTimeoutNs of %globaltimer, or kSyncMaxPolls
// polls) and reports whether it succeeded, so a missing producer ends in an
// error status, never in a hang.
#pragma once

#include <stdint.h>

namespace moe {

constexpr uint64_t kSyncTimeoutNs = 1000000000ull;  // one second
constexpr uint32_t kSyncMaxPolls = 1u << 24;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint64_t tagged_word(uint32_t tag, uint32_t value) {
  return ((uint64_t)tag << 32) | value;
}

__device__ __forceinline__ bool has_tag(uint64_t word, uint32_t tag) {
  return (uint32_t)(word >> 32) == tag;
}

__device__ __forceinline__ void store_tagged(uint64_t* p, uint32_t tag, uint32_t value) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(tagged_word(tag, value))
               : "memory");
}

__device__ __forceinline__ uint64_t load_relaxed(const uint64_t* p) {
  uint64_t x;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(x) : "l"(p) : "memory");
  return x;
}

__device__ __forceinline__ uint32_t load_relaxed(const uint32_t* p) {
  uint32_t x;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(x) : "l"(p) : "memory");
  return x;
}

__device__ __forceinline__ void add_relaxed(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Waits (one thread) until the counter *p reaches `target`; false once the
// time or poll limit is reached. A counter only says that waiting on the
// tagged words themselves is now worthwhile: the words are still checked.
__device__ __forceinline__ bool wait_count(const uint32_t* p, uint32_t target) {
  if (load_relaxed(p) >= target) return true;
  const uint64_t t0 = global_ns();
  uint32_t polls = 0;
  do {
    if (++polls > kSyncMaxPolls || global_ns() - t0 > kSyncTimeoutNs) return false;
    __nanosleep(32);
  } while (load_relaxed(p) < target);
  return true;
}

// Waits (one thread) until *p carries `tag`, then returns true with the value
// in `value`; returns false once the time or poll limit is reached.
__device__ __forceinline__ bool wait_tagged(const uint64_t* p, uint32_t tag, uint32_t& value) {
  uint64_t x = load_relaxed(p);
  if (!has_tag(x, tag)) {
    const uint64_t t0 = global_ns();
    uint32_t polls = 0;
    do {
      if (++polls > kSyncMaxPolls || global_ns() - t0 > kSyncTimeoutNs) return false;
      __nanosleep(64);
      x = load_relaxed(p);
    } while (!has_tag(x, tag));
  }
  value = (uint32_t)x;
  return true;
}

}  // namespace moe
