/*
 * sdcp_oracle_commit.c - plain CPU oracle of the steps around the SDCP verifier's
 * acceptance: the verifier's HMAC-SHA-256 random values, the committed-prefix digest
 * chain, truncation of the emitted tokens, and speculation control.
 *
 * TEST INFRASTRUCTURE, like sdcp_oracle.c: only tests/, __graft_entry__.smoke() and
 * bench.py load it.  It shares no code, header or constant with the CUDA path.
 *
 * Definitions followed (IETF draft-li-mlc-inference-acceleration-00, "Speculative
 * Decoding Coordination Protocol (SDCP) for Distributed Inference with Multi-Level
 * Caches"):
 *   Section 4.2: d[0] = SHA-256("SDCP-PREFIX-1" || 0x00 || contract_digest || uint32(P)
 *     || uint32(t[0]) || ... || uint32(t[P-1])), d[k] = SHA-256(d[k-1] || uint32(o[k]));
 *     uint32 is four octets, network byte order.
 *   Section 4.1: contract_digest = SHA-256("SDCP-CONTRACT-1" || 0x00 || cbor(contract)).
 *   Section 6.3, step "Acceptance": the emitted tokens are truncated after the first
 *     stop token and at max_new; step "Commit": n and d[n] are updated.
 *   Section 6.4, last paragraph: each random value is HMAC-SHA-256 keyed with the seed as
 *     eight octets (network byte order) over "SDCP-VERIFY-1" || 0x00 || session ||
 *     uint32(round) || uint32(i) || uint8(purpose); the first 53 bits / 2^53.
 *   Section 6.5: m_cap, low rounds, the counters c, g, j and the fallback ladder.
 * SHA-256: FIPS 180-4 (the algorithm of RFC 6234), its constants derived here from their
 * definition (fractional parts of square and cube roots of the first primes).  HMAC:
 * RFC 2104 with a 64-octet block.
 *
 * Readings where the pages leave a step open (listed in the design notes):
 *   - the index i of a random value is the 1-based position of the pages (p[1..M+1]): the
 *     acceptance test of 0-based position k uses i = k + 1, and the additional token drawn
 *     after a accepted tokens uses i = a + 1;
 *   - a stop token is itself emitted (truncation is after it); with n tokens committed
 *     before the round, at most max_new - n tokens are emitted (none once n >= max_new);
 *   - the round ends generation ("finish") when a stop token was emitted or n reaches
 *     max_new; the action is then finish, the counters c and g still follow the round's
 *     low / not-low outcome, and no ladder entry is applied;
 *   - after a round that is not low, m_cap grows by m_restore (0: never), capped at m_max
 *     ("restore gradually, for example by one per round");
 *   - self_decode is permitted when self_load is present (<= 100) and the verifier's load
 *     does not exceed it.
 */
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* ---------------------------------------------------------------------------------- */
/* SHA-256 (FIPS 180-4)                                                                 */
/* ---------------------------------------------------------------------------------- */
static uint32_t K256[64], H256[8];
static int sha_ready = 0;

/* floor(n^(1/e)) of an integer n < 2^110, by bisection (e = 2 or 3; the root is below
   2^40, so no product overflows 128 bits). */
static unsigned __int128 iroot(unsigned __int128 n, int e) {
  unsigned __int128 lo = 0, hi = (unsigned __int128)1 << 40;
  while (lo < hi) {
    unsigned __int128 mid = lo + (hi - lo + 1) / 2;
    unsigned __int128 p = mid * mid;
    if (e == 3) p *= mid;
    if (p <= n) lo = mid; else hi = mid - 1;
  }
  return lo;
}

/* The first 32 bits of the fractional part of the e-th root of p: floor(p^(1/e) * 2^32)
   mod 2^32 = floor((p * 2^(32 e))^(1/e)) mod 2^32. */
static uint32_t frac_root_bits(unsigned p, int e) {
  unsigned __int128 n = (unsigned __int128)p << (32 * e);
  return (uint32_t)iroot(n, e);
}

static void sha_init_constants(void) {
  if (sha_ready) return;
  unsigned primes[64];
  int np = 0;
  for (unsigned c = 2; np < 64; ++c) {
    int is_p = 1;
    for (unsigned d = 2; d * d <= c; ++d) if (c % d == 0) { is_p = 0; break; }
    if (is_p) primes[np++] = c;
  }
  for (int i = 0; i < 64; ++i) K256[i] = frac_root_bits(primes[i], 3); /* cube roots */
  for (int i = 0; i < 8; ++i) H256[i] = frac_root_bits(primes[i], 2);  /* square roots */
  sha_ready = 1;
}

/* Formed once when the library is loaded, before any OpenMP thread can use them. */
__attribute__((constructor)) static void sha_constants_at_load(void) { sha_init_constants(); }

static uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

/* One compression of a 64-octet block into the state h. */
static void sha_compress(uint32_t h[8], const uint8_t block[64]) {
  uint32_t w[64];
  for (int t = 0; t < 16; ++t)
    w[t] = ((uint32_t)block[4 * t] << 24) | ((uint32_t)block[4 * t + 1] << 16) |
           ((uint32_t)block[4 * t + 2] << 8) | (uint32_t)block[4 * t + 3];
  for (int t = 16; t < 64; ++t) {
    uint32_t s0 = rotr(w[t - 15], 7) ^ rotr(w[t - 15], 18) ^ (w[t - 15] >> 3);
    uint32_t s1 = rotr(w[t - 2], 17) ^ rotr(w[t - 2], 19) ^ (w[t - 2] >> 10);
    w[t] = w[t - 16] + s0 + w[t - 7] + s1;
  }
  uint32_t a = h[0], b = h[1], c = h[2], d = h[3], e = h[4], f = h[5], g = h[6], k = h[7];
  for (int t = 0; t < 64; ++t) {
    uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
    uint32_t ch = (e & f) ^ (~e & g);
    uint32_t t1 = k + S1 + ch + K256[t] + w[t];
    uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
    uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
    uint32_t t2 = S0 + maj;
    k = g; g = f; f = e; e = d + t1; d = c; c = b; b = a; a = t1 + t2;
  }
  h[0] += a; h[1] += b; h[2] += c; h[3] += d; h[4] += e; h[5] += f; h[6] += g; h[7] += k;
}

/* SHA-256 of msg[0..len) into out[32]: the message, a 1 bit, zeros, and its bit length as
   a 64-bit big-endian number, in 64-octet blocks. */
void oracle_sha256(const uint8_t* msg, size_t len, uint8_t out[32]) {
  sha_init_constants();
  uint32_t h[8];
  memcpy(h, H256, sizeof h);
  size_t full = len / 64;
  for (size_t i = 0; i < full; ++i) sha_compress(h, msg + 64 * i);
  uint8_t tail[128];
  size_t rem = len - 64 * full;
  memset(tail, 0, sizeof tail);
  memcpy(tail, msg + 64 * full, rem);
  tail[rem] = 0x80;
  size_t nb = (rem + 1 + 8 <= 64) ? 1 : 2;
  uint64_t bits = (uint64_t)len * 8u;
  for (int i = 0; i < 8; ++i) tail[64 * nb - 1 - i] = (uint8_t)(bits >> (8 * i));
  for (size_t i = 0; i < nb; ++i) sha_compress(h, tail + 64 * i);
  for (int i = 0; i < 8; ++i) {
    out[4 * i] = (uint8_t)(h[i] >> 24); out[4 * i + 1] = (uint8_t)(h[i] >> 16);
    out[4 * i + 2] = (uint8_t)(h[i] >> 8); out[4 * i + 3] = (uint8_t)h[i];
  }
}

/* HMAC-SHA-256 (RFC 2104): H((K ^ opad) || H((K ^ ipad) || msg)), K zero-padded to 64
   octets (a longer key is hashed first). */
void oracle_hmac_sha256(const uint8_t* key, size_t klen, const uint8_t* msg, size_t mlen,
                        uint8_t out[32]) {
  uint8_t k0[64];
  memset(k0, 0, sizeof k0);
  if (klen > 64) oracle_sha256(key, klen, k0);
  else memcpy(k0, key, klen);
  uint8_t buf[64 + 256];
  uint8_t inner[32];
  if (mlen > 256) mlen = 256; /* the callers here hash short messages only */
  for (int i = 0; i < 64; ++i) buf[i] = k0[i] ^ 0x36;
  memcpy(buf + 64, msg, mlen);
  oracle_sha256(buf, 64 + mlen, inner);
  for (int i = 0; i < 64; ++i) buf[i] = k0[i] ^ 0x5c;
  memcpy(buf + 64, inner, 32);
  oracle_sha256(buf, 96, out);
}

static void put_u32(uint8_t* p, uint32_t v) {
  p[0] = (uint8_t)(v >> 24); p[1] = (uint8_t)(v >> 16); p[2] = (uint8_t)(v >> 8); p[3] = (uint8_t)v;
}

/* ---------------------------------------------------------------------------------- */
/* The verifier's random values (Section 6.4, last paragraph).                         */
/* ---------------------------------------------------------------------------------- */
double oracle_hmac_uniform(uint64_t seed, const uint8_t session[16], uint32_t round, uint32_t i,
                           uint32_t purpose) {
  uint8_t key[8];
  for (int b = 0; b < 8; ++b) key[b] = (uint8_t)(seed >> (56 - 8 * b));
  static const char label[] = "SDCP-VERIFY-1";
  uint8_t msg[13 + 1 + 16 + 4 + 4 + 1];
  memcpy(msg, label, 13);
  msg[13] = 0x00;
  memcpy(msg + 14, session, 16);
  put_u32(msg + 30, round);
  put_u32(msg + 34, i);
  msg[38] = (uint8_t)purpose;
  uint8_t mac[32];
  oracle_hmac_sha256(key, 8, msg, sizeof msg, mac);
  uint64_t top = 0;
  for (int b = 0; b < 8; ++b) top = (top << 8) | mac[b];
  return (double)(top >> 11) * (1.0 / 9007199254740992.0); /* 2^53 */
}

/* ---------------------------------------------------------------------------------- */
/* Digests (Sections 4.1 and 4.2).                                                      */
/* ---------------------------------------------------------------------------------- */
void oracle_contract_digest(const uint8_t* cbor, size_t len, uint8_t out[32]) {
  uint8_t buf[16 + 4096];
  if (len > 4096) len = 4096;
  memcpy(buf, "SDCP-CONTRACT-1", 15);
  buf[15] = 0x00;
  memcpy(buf + 16, cbor, len);
  oracle_sha256(buf, 16 + len, out);
}

/* d[0] of a prompt t[0..P). */
void oracle_prefix_digest(const uint8_t contract_digest[32], const uint32_t* prompt, uint32_t P,
                          uint8_t out[32]) {
  size_t len = 14 + 32 + 4 + 4 * (size_t)P;
  uint8_t stackbuf[1024];
  uint8_t* buf = stackbuf;
  if (len > sizeof stackbuf) return; /* the callers here use short prompts */
  memcpy(buf, "SDCP-PREFIX-1", 13);
  buf[13] = 0x00;
  memcpy(buf + 14, contract_digest, 32);
  put_u32(buf + 46, P);
  for (uint32_t k = 0; k < P; ++k) put_u32(buf + 50 + 4 * k, prompt[k]);
  oracle_sha256(buf, len, out);
}

/* d[n + m] from d[n] and the tokens o[n+1 .. n+m], one link at a time. */
void oracle_digest_extend(const uint8_t d[32], const int32_t* tokens, int32_t m, uint8_t out[32]) {
  uint8_t cur[32], buf[36];
  memcpy(cur, d, 32);
  for (int32_t k = 0; k < m; ++k) {
    memcpy(buf, cur, 32);
    put_u32(buf + 32, (uint32_t)tokens[k]);
    oracle_sha256(buf, 36, cur);
  }
  memcpy(out, cur, 32);
}

/* ---------------------------------------------------------------------------------- */
/* Truncation, commit and control of one session's round (Sections 6.3, 6.5).          */
/* ---------------------------------------------------------------------------------- */
enum { ACT_CONTINUE = 0, ACT_REDUCE = 1, ACT_SWITCH = 2, ACT_SELF_DECODE = 3, ACT_FINISH = 4,
       ACT_FAIL = 5 };

typedef struct {           /* contract terms (Section 4.1) */
  uint32_t max_new, stop_offset, stop_count, m_max;
  uint32_t low_rounds, low_ratio, self_load, fallback_len;
  uint8_t fallback[8];
  uint32_t m_restore, pad;
} orc_commit_params;

typedef struct {           /* the verifier's per-session state */
  uint8_t digest[32];
  uint32_t committed, c, g, j, m_cap, pad[3];
} orc_session_state;

/*
 * One round of session b after acceptance: emitted = out_tokens[0 .. n_out) (a accepted
 * plus the additional token), M proposed.  Truncates (in place: n_out, and the dropped
 * slots set to -1), commits (state->committed, state->digest), and runs control
 * (state->c, g, j, m_cap).  Returns the action.
 */
int32_t oracle_commit_round(const orc_commit_params* cp, const uint32_t* stop_tokens,
                            orc_session_state* st, int32_t a, int32_t M, int32_t* n_out,
                            int32_t* out_tokens, uint32_t load) {
  int32_t n = *n_out;
  int finished = 0;
  for (int32_t k = 0; k < n; ++k) {
    int is_stop = 0;
    for (uint32_t s = 0; s < cp->stop_count; ++s)
      if ((uint32_t)out_tokens[k] == stop_tokens[cp->stop_offset + s]) is_stop = 1;
    if (is_stop) { n = k + 1; finished = 1; break; }
  }
  uint32_t room = (st->committed >= cp->max_new) ? 0u : cp->max_new - st->committed;
  if ((uint32_t)n >= room) { n = (int32_t)room; finished = 1; }
  for (int32_t k = n; k < *n_out; ++k) out_tokens[k] = -1;
  *n_out = n;
  oracle_digest_extend(st->digest, out_tokens, n, st->digest);
  st->committed += (uint32_t)n;

  /* Section 6.5.2: is the round low?  (The contract requires low_rounds >= 1 and at most
     eight ladder entries here; other values are read as the nearest valid one.) */
  const uint32_t R = cp->low_rounds < 1 ? 1 : cp->low_rounds;
  const uint32_t nfb = cp->fallback_len > 8 ? 8 : cp->fallback_len;
  int low = (cp->low_ratio != 0) ? ((uint64_t)100 * (uint32_t)a < (uint64_t)cp->low_ratio * (uint32_t)M)
                                 : (a == 0);
  if (low) { st->c += 1; st->g = 0; }
  else {
    st->c = 0; st->g += 1;
    if (st->g >= R) st->j = 0;
    uint32_t mc = st->m_cap + cp->m_restore;
    st->m_cap = mc > cp->m_max ? cp->m_max : mc;
  }
  if (finished) return ACT_FINISH;
  int32_t action = ACT_CONTINUE;
  if (st->c >= R) {
    action = ACT_FAIL; /* unless an entry remains */
    while (st->j < nfb) {
      uint8_t e = cp->fallback[st->j];
      st->j += 1;
      if (e == ACT_SELF_DECODE && !(cp->self_load <= 100 && load <= cp->self_load)) continue;
      action = e;
      break;
    }
    st->c = 0;
    if (action == ACT_REDUCE) st->m_cap = (st->m_cap / 2 > 1) ? st->m_cap / 2 : 1;
  }
  return action;
}
