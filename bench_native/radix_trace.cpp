// Replay of a chat-like request trace through the prefix index's C ABI, with
// no Python in the loop: the native throughput of pkv_radix_*.
//
// Trace ("PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", section 03:
// many requests over a few shared prompts): 64 system prompts of 1,000 token
// ids, each request one of them plus a question of 10..200 ids, 16-token
// blocks, a pool of 8,192 blocks so that eviction runs.  Every request does
// match, alloc (its new blocks), insert, release and frees its partial last
// block.  Token ids come from std::mt19937_64 (seed 0), whose output the C++
// standard fixes, so the trace is the same on every platform.
//
// Usage: radix_trace [num_requests]; prints one JSON object.
#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <random>
#include <vector>

#include "pkv.h"

int main(int argc, char** argv) {
  const int n = argc > 1 ? std::atoi(argv[1]) : 20000;
  const int bs = 16, pool = 8192;
  std::mt19937_64 rng(0);
  std::vector<std::vector<int32_t>> prompts(64);
  for (auto& p : prompts) {
    p.resize(1000);
    for (auto& t : p) t = (int32_t)(rng() % 32000);
  }
  std::vector<std::vector<int32_t>> reqs((size_t)(n > 0 ? n : 0));
  for (auto& r : reqs) {
    r = prompts[rng() % 64];
    const int q = 10 + (int)(rng() % 191);
    for (int i = 0; i < q; ++i) r.push_back((int32_t)(rng() % 32000));
  }
  pkv_radix_index* x = nullptr;
  if (pkv_radix_create(bs, pool, &x) != PKV_OK) return 1;
  std::vector<int32_t> matched(128), table(128), released(128);
  long long hit = 0, total = 0, refused = 0;
  const auto t0 = std::chrono::steady_clock::now();
  for (const auto& r : reqs) {
    const int len = (int)r.size();
    int32_t m = 0;
    if (pkv_radix_match(x, r.data(), len, matched.data(), (int32_t)matched.size(), &m) != PKV_OK)
      return 1;
    const int have = m / bs, need = (len + bs - 1) / bs - have;
    for (int i = 0; i < have; ++i) table[i] = matched[i];
    if (pkv_radix_alloc(x, need, table.data() + have) != PKV_OK) {
      pkv_radix_release(x, r.data(), m);
      ++refused;
      continue;
    }
    int32_t nrel = 0;
    if (pkv_radix_insert(x, r.data(), len, table.data(), released.data(), &nrel) != PKV_OK) return 1;
    if (pkv_radix_release(x, r.data(), m) != PKV_OK) return 1;
    if (len % bs && pkv_radix_free(x, table.data() + have + need - 1, 1) != PKV_OK) return 1;
    hit += m;
    total += len;
  }
  const double dt =
      std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
  pkv_radix_destroy(x);
  std::printf(
      "{\"requests\": %d, \"requests_per_s\": %.1f, \"us_per_request\": %.3f, "
      "\"cached_token_frac\": %.4f, \"refused\": %lld}\n",
      n, n / dt, dt / (n > 0 ? n : 1) * 1e6, total ? (double)hit / (double)total : 0.0, refused);
  return 0;
}
