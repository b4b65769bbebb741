// Host-side layout builder: prime sequence, segment offsets, odd multipliers.
//
// Pages cited by title:
//   [P-V41] "DeepSeek-V4.1 模型结构（5）：记忆，Engram"
//   [P-O1]  "条件记忆：DeepSeek V4.1 Engram 如何用 O(1) 查表换掉一层计算"
//   [P-DS4] "ds4.c 学习笔记" -- glossary entry "Engram"
#include <stdint.h>

#include <cstring>

#include "engram_internal.h"

namespace engram {
namespace {

using u64 = uint64_t;
using u128 = unsigned __int128;

u64 mulmod(u64 a, u64 b, u64 m) { return static_cast<u64>((static_cast<u128>(a) * b) % m); }

u64 powmod(u64 a, u64 e, u64 m) {
  u64 r = 1 % m;
  a %= m;
  while (e) {
    if (e & 1) r = mulmod(r, a, m);
    a = mulmod(a, a, m);
    e >>= 1;
  }
  return r;
}

// Deterministic Miller-Rabin: the first twelve primes as bases decide every
// n < 3.3e24, hence every 64-bit n (Sorenson & Webster, Math. Comp. 2017).
// [P-O1] §2.2 names a deterministic Miller-Rabin test for the prime search.
bool is_prime_u64(u64 n) {
  static const u64 bases[] = {2, 3, 5, 7, 11, 13, 17, 19, 23, 29, 31, 37};
  if (n < 2) return false;
  for (u64 p : bases) {
    if (n % p == 0) return n == p;
  }
  u64 d = n - 1;
  int s = 0;
  while ((d & 1) == 0) {
    d >>= 1;
    ++s;
  }
  for (u64 a : bases) {
    u64 x = powmod(a, d, n);
    if (x == 1 || x == n - 1) continue;
    bool composite = true;
    for (int r = 1; r < s; ++r) {
      x = mulmod(x, x, n);
      if (x == n - 1) {
        composite = false;
        break;
      }
    }
    if (composite) return false;
  }
  return true;
}

// SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): advance the state by the
// golden gamma, then a xor-shift-multiply finaliser.
struct SplitMix64 {
  u64 state;
  u64 next() {
    state += 0x9E3779B97F4A7C15ull;
    u64 z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }
};

constexpr u64 kInt64Max = 0x7FFFFFFFFFFFFFFFull;

}  // namespace
}  // namespace engram

extern "C" int engram_build_layout(const engram_layout_params* p, engram_layout* out) {
  using namespace engram;
  if (p == nullptr || out == nullptr) return fail(ENGRAM_E_INVALID, "null argument");
  const int64_t V = p->vocab_compressed;
  if (V < 2) return fail(ENGRAM_E_INVALID, "compressed vocabulary %lld < 2", (long long)V);
  // [P-V41] under eq. (H): the code checks the compressed vocabulary at start
  // and refuses to run when it differs -- every multiplier depends on it.
  if (p->expected_vocab != 0 && p->expected_vocab != V)
    return fail(ENGRAM_E_VOCAB, "compressed vocabulary %lld != expected %lld", (long long)V,
                (long long)p->expected_vocab);
  if (p->n_layers < 1 || p->n_layers > ENGRAM_MAX_LAYERS)
    return fail(ENGRAM_E_INVALID, "n_layers %d not in [1, %d]", p->n_layers, ENGRAM_MAX_LAYERS);
  if (p->max_ngram < 2 || p->max_ngram > ENGRAM_MAX_NGRAM)
    return fail(ENGRAM_E_SHAPE, "max_ngram %d not in [2, %d]", p->max_ngram, ENGRAM_MAX_NGRAM);
  if (p->n_heads < 1) return fail(ENGRAM_E_INVALID, "n_heads %d < 1", p->n_heads);
  const int n_cols = (p->max_ngram - 1) * p->n_heads;
  if (n_cols > ENGRAM_MAX_COLS)
    return fail(ENGRAM_E_SHAPE, "(max_ngram-1)*n_heads = %d > %d", n_cols, ENGRAM_MAX_COLS);
  if (p->head_dim != ENGRAM_HEAD_DIM)
    return fail(ENGRAM_E_SHAPE, "head_dim %d: only 256-dim E4M3 rows are supported", p->head_dim);
  if (p->pad_id < 0 || p->pad_id >= V)
    return fail(ENGRAM_E_INVALID, "pad_id %d is not a compressed id in [0, %lld)", p->pad_id,
                (long long)V);
  if (p->base_rows < 0) return fail(ENGRAM_E_INVALID, "base_rows < 0");

  engram_layout L;
  std::memset(&L, 0, sizeof(L));
  L.vocab_compressed = V;
  L.base_rows = p->base_rows;
  L.n_layers = p->n_layers;
  L.max_ngram = p->max_ngram;
  L.n_heads = p->n_heads;
  L.n_cols = n_cols;
  L.head_dim = p->head_dim;
  L.pad_id = p->pad_id;

  // [P-V41] §"一层只有一张表", [P-O1] §2.2: one ascending prime sequence
  // starting above engram_vocab_size, consumed in (layer, order, head) order,
  // one prime per column, never reused.
  u64 cand = static_cast<u64>(p->base_rows);
  const u64 half = (kInt64Max / static_cast<u64>(V)) / 2;
  for (int l = 0; l < p->n_layers; ++l) {
    L.layer_ids[l] = p->layer_ids[l];
    int64_t acc = 0;
    for (int j = 0; j < n_cols; ++j) {
      do {
        ++cand;
      } while (!is_prime_u64(cand));
      L.primes[l][j] = static_cast<int64_t>(cand);
      L.offsets[l][j] = acc;  // [P-O1] §2.2: offsets are the cumulative sum
      L.reciprocal[l][j] = ~0ull / cand;
      acc += static_cast<int64_t>(cand);
      if (acc >= (int64_t(1) << 31))
        return fail(ENGRAM_E_RANGE, "layer %d table would have %lld >= 2^31 rows", l,
                    (long long)acc);
    }
    L.total_rows[l] = acc;
    // Multipliers: odd and bounded so that (V-1) * m fits in int64
    // ([P-V41] under eq. (H); [P-O1] §4.3: seed 10007 * layer_id,
    // bound int64max // V // 2).
    if (p->use_multiplier_override) {
      for (int i = 0; i < p->max_ngram; ++i) {
        int64_t m = p->multiplier_override[l][i];
        if (m <= 0 || (m & 1) == 0 || static_cast<u64>(m) > kInt64Max / static_cast<u64>(V - 1))
          return fail(ENGRAM_E_RANGE,
                      "override multiplier %lld (layer %d, i %d) must be odd and keep (V-1)*m in int64",
                      (long long)m, l, i);
        L.multipliers[l][i] = m;
      }
    } else {
      SplitMix64 rng{static_cast<u64>(10007) * static_cast<u64>(static_cast<int64_t>(p->layer_ids[l]))};
      for (int i = 0; i < p->max_ngram; ++i) {
        u64 r = rng.next() % half;
        L.multipliers[l][i] = static_cast<int64_t>(2 * r + 1);
      }
    }
  }
  *out = L;
  return ENGRAM_OK;
}
