// rope_table.cpp -- host-side RoPE cos/sin table in fp64, stored as fp32.
//
// gaudi-cookbook "MiMo-V2.6-Flash on Gaudi 2", section "The RoPE fix for
// large positions": fp32 cos/sin of angles past about 1.5e5 rad are wrong
// (the fastest rotary frequency's angle equals the position in radians), so
// the table is evaluated on the CPU in float64 and only the results are
// rounded to fp32.  colibri "MiMo-V2.6", "What the engine implements": the
// rotation covers the first 64 of 192 dims, i.e. 32 frequencies
// inv_freq_i = theta^(-2i/64).
#include <cmath>
#include <cstdint>
#include <thread>
#include <vector>

namespace kvr {

void rope_table_fill(double theta, int64_t max_pos, float *out, int nthreads) {
  double inv_freq[32];
  for (int i = 0; i < 32; ++i) inv_freq[i] = std::pow(theta, -(2.0 * i) / 64.0);
  auto work = [&](int64_t lo, int64_t hi) {
    for (int64_t p = lo; p < hi; ++p) {
      float *row = out + p * 64;
      for (int i = 0; i < 32; ++i) {
        const double a = static_cast<double>(p) * inv_freq[i];
        row[2 * i] = static_cast<float>(std::cos(a));
        row[2 * i + 1] = static_cast<float>(std::sin(a));
      }
    }
  };
  if (nthreads <= 0) nthreads = static_cast<int>(std::thread::hardware_concurrency());
  if (nthreads < 1) nthreads = 1;
  if (max_pos < 4096 || nthreads == 1) {
    work(0, max_pos);
    return;
  }
  std::vector<std::thread> pool;
  const int64_t per = (max_pos + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    const int64_t lo = t * per, hi = std::min<int64_t>(max_pos, lo + per);
    if (lo >= hi) break;
    pool.emplace_back(work, lo, hi);
  }
  for (auto &th : pool) th.join();
}

}  // namespace kvr
