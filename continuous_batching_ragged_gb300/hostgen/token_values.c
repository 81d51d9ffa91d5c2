/* Seeded synthetic token values on the host CPU (input generation only).
 *
 * A plain C restatement of the value definition that workloads.py documents
 * and implements in numpy: Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3", SC'11) on the counter
 * (head * A + dim, position, seq_id, kind << 16 | layer) keyed by the seed,
 * then an exact Irwin-Hall(8) normal approximation, then (for bf16) rounding
 * to the nearest bf16, ties to even.  It exists because the numpy version
 * runs one full Philox per value and is too slow for the oracle's full-size
 * inputs (hundreds of millions of values); tests pin it bit for bit to the
 * numpy version.  It holds none of the attention or scheduling arithmetic and
 * shares nothing with the CUDA library.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

static void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)PHILOX_M0 * c[0];
    const uint64_t p1 = (uint64_t)PHILOX_M1 * c[2];
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
    k0 += PHILOX_W0;
    k1 += PHILOX_W1;
  }
}

static uint32_t f32_bits(float x) {
  uint32_t u;
  memcpy(&u, &x, sizeof u);
  return u;
}

static float bits_f32(uint32_t u) {
  float x;
  memcpy(&x, &u, sizeof x);
  return x;
}

/* out[i][j][d] for positions[i], heads[j], d < head_dim (fp32 holding the
 * dtype's value).  bf16 != 0 rounds each value to bf16. */
void cbv_token_values(uint64_t seed, uint32_t kind, uint32_t layer, uint32_t seq_id,
                      const uint32_t* positions, int64_t n_pos, const uint32_t* heads, int32_t n_heads,
                      int32_t head_dim, int32_t bf16, float* out) {
  const float scale = (float)(sqrt(1.5) / 131072.0);
  const uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  const uint32_t c3 = ((kind & 0xFFFFu) << 16) | (layer & 0xFFFFu);
  for (int64_t i = 0; i < n_pos; ++i) {
    for (int32_t j = 0; j < n_heads; ++j) {
      float* o = out + ((size_t)i * n_heads + j) * head_dim;
      for (int32_t d = 0; d < head_dim; ++d) {
        uint32_t c[4] = {heads[j] * (uint32_t)head_dim + (uint32_t)d, positions[i], seq_id, c3};
        philox4x32_10(c, k0, k1);
        int64_t s = 0;
        for (int w = 0; w < 4; ++w) s += (int64_t)(c[w] & 0xFFFFu) + (int64_t)(c[w] >> 16);
        const int64_t s2 = 2 * s - 8 * 65535;
        float x = (float)s2 * scale;
        if (bf16) {
          const uint64_t u = f32_bits(x);
          const uint64_t r = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
          x = bits_f32((uint32_t)(r << 16));
        }
        o[d] = x;
      }
    }
  }
}
