// Seeded synthetic input generator for the MoE layer workloads.
//
// This file holds no arithmetic of the MoE layer itself: it only turns
// (seed, tensor id, element index) into a number.  Both the CPU oracle and
// the CUDA path receive the bytes it writes, so they always see identical
// inputs.
//
// Definition (counter based, so any sub-range can be generated on its own):
//   mix64(z)   = the splitmix64 finaliser (Steele, Lea, Flood, "Fast
//                splittable pseudorandom number generators", OOPSLA 2014):
//                z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
//                z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31.
//   base       = mix64(seed + 0x9E3779B97F4A7C15) ^ (tensor_id * 0xD1B54A32D192ED03)
//   word(c)    = mix64(base + (c + 1) * 0x9E3779B97F4A7C15)
//   u1(i)      = ((word(2i) >> 11) + 1) * 2^-53        in (0, 1]
//   u2(i)      = (word(2i+1) >> 11) * 2^-53            in [0, 1)
//   normal(i)  = sqrt(-2 ln u1) * cos(2 pi u2)         (Box-Muller, cosine branch)
//   value(i)   = mean + std * normal(i), in double, rounded to float (RNE),
//                and for bf16 storage rounded once more float -> bf16 (RNE).
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

inline uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

inline uint64_t stream_base(uint64_t seed, uint64_t tid) {
  return mix64(seed + kGolden) ^ (tid * 0xD1B54A32D192ED03ull);
}

inline double normal_at(uint64_t base, uint64_t i) {
  const uint64_t w1 = mix64(base + (2 * i + 1) * kGolden);
  const uint64_t w2 = mix64(base + (2 * i + 2) * kGolden);
  const double u1 = (double)((w1 >> 11) + 1) * 0x1.0p-53;
  const double u2 = (double)(w2 >> 11) * 0x1.0p-53;
  return std::sqrt(-2.0 * std::log(u1)) * std::cos(6.283185307179586476925286766559 * u2);
}

inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

template <typename Fn>
void parallel_for(int64_t n, int nthreads, Fn fn) {
  if (nthreads <= 1 || n < (1 << 16)) {
    fn(0, n);
    return;
  }
  std::vector<std::thread> th;
  const int64_t chunk = (n + nthreads - 1) / nthreads;
  for (int w = 0; w < nthreads; ++w) {
    const int64_t lo = w * chunk, hi = std::min<int64_t>(n, lo + chunk);
    if (lo >= hi) break;
    th.emplace_back([=] { fn(lo, hi); });
  }
  for (auto& t : th) t.join();
}

int default_threads(int nthreads) {
  if (nthreads > 0) return nthreads;
  unsigned hc = std::thread::hardware_concurrency();
  return hc ? (int)hc : 1;
}

}  // namespace

extern "C" {

// Writes n values, elements [start, start + n) of stream (seed, tensor_id), as bf16 bits.
void synth_normal_bf16(uint64_t seed, uint64_t tensor_id, uint64_t start, int64_t n, double mean,
                       double stdev, uint16_t* out, int nthreads) {
  const uint64_t base = stream_base(seed, tensor_id);
  parallel_for(n, default_threads(nthreads), [&](int64_t lo, int64_t hi) {
    for (int64_t i = lo; i < hi; ++i)
      out[i] = f32_to_bf16_rne((float)(mean + stdev * normal_at(base, start + (uint64_t)i)));
  });
}

// Same stream definition, stored as float32.
void synth_normal_f32(uint64_t seed, uint64_t tensor_id, uint64_t start, int64_t n, double mean,
                      double stdev, float* out, int nthreads) {
  const uint64_t base = stream_base(seed, tensor_id);
  parallel_for(n, default_threads(nthreads), [&](int64_t lo, int64_t hi) {
    for (int64_t i = lo; i < hi; ++i) out[i] = (float)(mean + stdev * normal_at(base, start + (uint64_t)i));
  });
}

// Raw 64-bit words of the stream (used by tests of the generator itself).
void synth_words(uint64_t seed, uint64_t tensor_id, uint64_t start, int64_t n, uint64_t* out) {
  const uint64_t base = stream_base(seed, tensor_id);
  for (int64_t i = 0; i < n; ++i) out[i] = mix64(base + (start + (uint64_t)i + 1) * kGolden);
}

}  // extern "C"
