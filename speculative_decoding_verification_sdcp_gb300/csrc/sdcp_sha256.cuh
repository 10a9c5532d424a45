// sdcp_sha256.cuh - SHA-256 on the GPU for the SDCP verifier: one compression per thread,
// the state in registers.  Used by the committed-prefix digest chain (SDCP draft Section
// 4.2) and by the verifier's HMAC-SHA-256 random values (Section 6.4, last paragraph).
//
// SHA-256 is FIPS 180-4 (the algorithm of RFC 6234): the round constants are the first 32
// bits of the fractional parts of the cube roots of the first 64 primes, the initial value
// those of the square roots of the first 8 primes.  HMAC is RFC 2104 with a 64-octet block.
#pragma once

#include <stdint.h>

namespace sdcp {

__device__ __forceinline__ uint32_t rotr32(uint32_t x, int n) { return __funnelshift_r(x, x, n); }

struct Sha256State {
  uint32_t h[8];
};

__device__ __forceinline__ Sha256State sha256_iv() {
  return Sha256State{{0x6a09e667u, 0xbb67ae85u, 0x3c6ef372u, 0xa54ff53au,
                      0x510e527fu, 0x9b05688cu, 0x1f83d9abu, 0x5be0cd19u}};
}

// One compression of the 16 big-endian words w of a block into s (FIPS 180-4, 6.2.2).
static __device__ __noinline__ Sha256State sha256_compress(Sha256State s, const uint32_t (&blk)[16]) {
  constexpr uint32_t K[64] = {
      0x428a2f98u, 0x71374491u, 0xb5c0fbcfu, 0xe9b5dba5u, 0x3956c25bu, 0x59f111f1u, 0x923f82a4u, 0xab1c5ed5u,
      0xd807aa98u, 0x12835b01u, 0x243185beu, 0x550c7dc3u, 0x72be5d74u, 0x80deb1feu, 0x9bdc06a7u, 0xc19bf174u,
      0xe49b69c1u, 0xefbe4786u, 0x0fc19dc6u, 0x240ca1ccu, 0x2de92c6fu, 0x4a7484aau, 0x5cb0a9dcu, 0x76f988dau,
      0x983e5152u, 0xa831c66du, 0xb00327c8u, 0xbf597fc7u, 0xc6e00bf3u, 0xd5a79147u, 0x06ca6351u, 0x14292967u,
      0x27b70a85u, 0x2e1b2138u, 0x4d2c6dfcu, 0x53380d13u, 0x650a7354u, 0x766a0abbu, 0x81c2c92eu, 0x92722c85u,
      0xa2bfe8a1u, 0xa81a664bu, 0xc24b8b70u, 0xc76c51a3u, 0xd192e819u, 0xd6990624u, 0xf40e3585u, 0x106aa070u,
      0x19a4c116u, 0x1e376c08u, 0x2748774cu, 0x34b0bcb5u, 0x391c0cb3u, 0x4ed8aa4au, 0x5b9cca4fu, 0x682e6ff3u,
      0x748f82eeu, 0x78a5636fu, 0x84c87814u, 0x8cc70208u, 0x90befffau, 0xa4506cebu, 0xbef9a3f7u, 0xc67178f2u};
  uint32_t w[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) w[t] = blk[t];
  uint32_t a = s.h[0], b = s.h[1], c = s.h[2], d = s.h[3], e = s.h[4], f = s.h[5], g = s.h[6], k = s.h[7];
#pragma unroll
  for (int t = 0; t < 64; ++t) {
    uint32_t wt;
    if (t < 16) {
      wt = w[t];
    } else {  // the message schedule, kept as a rolling window of 16 words
      const uint32_t w15 = w[(t - 15) & 15], w2 = w[(t - 2) & 15];
      const uint32_t s0 = rotr32(w15, 7) ^ rotr32(w15, 18) ^ (w15 >> 3);
      const uint32_t s1 = rotr32(w2, 17) ^ rotr32(w2, 19) ^ (w2 >> 10);
      wt = w[t & 15] + s0 + w[(t - 7) & 15] + s1;
      w[t & 15] = wt;
    }
    const uint32_t S1 = rotr32(e, 6) ^ rotr32(e, 11) ^ rotr32(e, 25);
    const uint32_t ch = (e & f) ^ (~e & g);
    const uint32_t t1 = k + S1 + ch + K[t] + wt;
    const uint32_t S0 = rotr32(a, 2) ^ rotr32(a, 13) ^ rotr32(a, 22);
    const uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
    k = g; g = f; f = e; e = d + t1; d = c; c = b; b = a; a = t1 + S0 + maj;
  }
  s.h[0] += a; s.h[1] += b; s.h[2] += c; s.h[3] += d; s.h[4] += e; s.h[5] += f; s.h[6] += g; s.h[7] += k;
  return s;
}

// One link of the committed-prefix digest chain: SHA-256(d || uint32(token)).  The 36
// octets fit one block: the digest's words (its octets in network order are the words of
// the state), the token, the padding bit and the length, 288 bits.
__device__ __forceinline__ Sha256State digest_link(const Sha256State& d, uint32_t token) {
  uint32_t blk[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) blk[i] = d.h[i];
  blk[8] = token;
  blk[9] = 0x80000000u;
#pragma unroll
  for (int i = 10; i < 15; ++i) blk[i] = 0u;
  blk[15] = 36u * 8u;
  return sha256_compress(sha256_iv(), blk);
}

// The verifier's random value by the draft's own derivation: HMAC-SHA-256 keyed with the
// 64-bit seed as eight octets in network order, over "SDCP-VERIFY-1" || 0x00 || session
// (16 octets) || uint32(round) || uint32(i) || uint8(purpose); the first 53 bits / 2^53.
// sid: the session identifier as four big-endian words.  i is the 1-based position.
static __device__ __noinline__ double hmac_uniform(uint64_t seed, const uint32_t (&sid)[4], uint32_t round,
                                            uint32_t i, uint32_t purpose) {
  // the key block (key zero-padded to 64 octets) xor ipad / opad, compressed once each
  uint32_t kb[16];
  const uint32_t k0 = (uint32_t)(seed >> 32), k1 = (uint32_t)seed;
#pragma unroll
  for (int t = 0; t < 16; ++t) kb[t] = (t == 0 ? k0 : (t == 1 ? k1 : 0u)) ^ 0x36363636u;
  const Sha256State si = sha256_compress(sha256_iv(), kb);
#pragma unroll
  for (int t = 0; t < 16; ++t) kb[t] = (t == 0 ? k0 : (t == 1 ? k1 : 0u)) ^ 0x5c5c5c5cu;
  const Sha256State so = sha256_compress(sha256_iv(), kb);
  // inner: the 39-octet message after the ipad block, padded; 103 octets in all
  uint32_t m[16];
  m[0] = 0x53444350u;  // "SDCP"
  m[1] = 0x2D564552u;  // "-VER"
  m[2] = 0x4946592Du;  // "IFY-"
  m[3] = 0x31000000u | (sid[0] >> 16);                       // "1", 0x00, session[0..1]
  m[4] = (sid[0] << 16) | (sid[1] >> 16);                    // session[2..5]
  m[5] = (sid[1] << 16) | (sid[2] >> 16);                    // session[6..9]
  m[6] = (sid[2] << 16) | (sid[3] >> 16);                    // session[10..13]
  m[7] = (sid[3] << 16) | (round >> 16);                     // session[14..15], round[0..1]
  m[8] = (round << 16) | (i >> 16);                          // round[2..3], i[0..1]
  m[9] = (i << 16) | ((purpose & 0xFFu) << 8) | 0x80u;       // i[2..3], purpose, padding bit
#pragma unroll
  for (int t = 10; t < 15; ++t) m[t] = 0u;
  m[15] = (64u + 39u) * 8u;
  const Sha256State inner = sha256_compress(si, m);
  // outer: the inner digest after the opad block, padded; 96 octets in all
#pragma unroll
  for (int t = 0; t < 8; ++t) m[t] = inner.h[t];
  m[8] = 0x80000000u;
#pragma unroll
  for (int t = 9; t < 15; ++t) m[t] = 0u;
  m[15] = (64u + 32u) * 8u;
  const Sha256State mac = sha256_compress(so, m);
  const unsigned long long bits = ((unsigned long long)mac.h[0] << 21) | (unsigned long long)(mac.h[1] >> 11);
  return (double)bits * 0x1.0p-53;
}

}  // namespace sdcp
