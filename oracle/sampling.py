"""Token selection beyond greedy: temperature / top-k sampling and the EOS stop.

The Kog monokernel tutorial ("How the monokernel removes launch overhead")
keeps LM-head sampling and the end-of-sequence check inside the one resident
kernel; the pages fix neither the sampler nor its random numbers.  Readings
taken here (the plainest that reproduce a softmax sample exactly):

* Sampling at temperature T > 0 draws token i with probability proportional
  to exp(l_i / T) over the candidate set: all tokens, or with top_k = k > 0
  the k largest logits (equal logits at the boundary: the lower index first).
  T == 0 is greedy argmax (lowest index among equal maxima).
* The draw is the Gumbel-max identity: the candidate with the largest
  l_i / T + g_i, g_i = -log(-log(u_i)), u_i uniform on (0, 1), is a sample
  from that softmax (Gumbel 1954; e.g. Maddison, Tarlow, Minka, "A* Sampling",
  2014).  Equal perturbed scores go to the lower index.
* u_i comes from the counter-based generator Philox4x32-10 (Salmon, Moraes,
  Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC 2011): key
  (seed_lo, seed_hi), counter (i, pos, 0, 0) with pos the absolute position of
  the token being fed, first output word x; u = (2 * (x >> 9) + 1) * 2^-24,
  which is exact in float32 and never 0 or 1.  Keying on the position makes a
  decode split over several calls draw the same numbers as one call.
* EOS: the step whose selected token equals eos_id is the last one; that
  token is emitted and decoding stops.

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""
import numpy as np

from . import llama

M0, M1 = np.uint64(0xD2511F53), np.uint64(0xCD9E8D57)   # Philox4x32 round multipliers
W0, W1 = np.uint32(0x9E3779B9), np.uint32(0xBB67AE85)   # key schedule (Weyl) increments
MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(counter, key):
    """Philox4x32 with 10 rounds.  counter: uint32 [..., 4]; key: uint32 [2]
    (or [..., 2]).  Returns uint32 [..., 4].

    One round: (hi0, lo0) = M0 * c0, (hi1, lo1) = M1 * c2 (64-bit products);
    c <- (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0).  The key is bumped by
    (W0, W1) between rounds."""
    c = np.asarray(counter, np.uint32).astype(np.uint64)
    k = np.broadcast_to(np.asarray(key, np.uint32), c.shape[:-1] + (2,)).astype(np.uint32)
    k0, k1 = k[..., 0].copy(), k[..., 1].copy()
    c0, c1, c2, c3 = (c[..., j] for j in range(4))
    for r in range(10):
        if r:
            k0 = (k0 + W0).astype(np.uint32)
            k1 = (k1 + W1).astype(np.uint32)
        p0 = M0 * c0
        p1 = M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0.astype(np.uint64), lo1, hi0 ^ c3 ^ k1.astype(np.uint64), lo0)
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def uniforms(n, pos, seed):
    """u_i for tokens i = 0..n-1 at position pos (float64, exact float32 values)."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint32)
    ctr = np.zeros((n, 4), np.uint32)
    ctr[:, 0] = np.arange(n, dtype=np.uint32)
    ctr[:, 1] = np.uint32(pos)
    x = philox4x32_10(ctr, key)[:, 0]
    return ((x >> np.uint32(9)).astype(np.float64) * 2.0 + 1.0) * 2.0 ** -24


def candidates(logits, top_k):
    """Indices of the candidate set: all tokens, or the top_k largest logits
    (ties at the boundary: lower index first), in ascending index order."""
    logits = np.asarray(logits, np.float64)
    if np.isnan(logits).any():
        raise ValueError("NaN logit")
    n = len(logits)
    if top_k <= 0 or top_k >= n:
        return np.arange(n)
    order = np.lexsort((np.arange(n), -logits))   # by value descending, then index ascending
    return np.sort(order[:top_k])


def perturbed(logits, idx, temperature, pos, seed):
    """l_i / T + g_i for the candidates idx (float64)."""
    u = uniforms(len(logits), pos, seed)[idx]
    return np.asarray(logits, np.float64)[idx] / temperature - np.log(-np.log(u))


def select(logits, temperature, top_k, pos, seed):
    """The selected token: greedy for T == 0, else the Gumbel-max sample."""
    if temperature == 0:
        return llama.argmax_lowest(logits)
    idx = candidates(logits, top_k)
    z = perturbed(logits, idx, temperature, pos, seed)
    return int(idx[np.flatnonzero(z == z.max())[0]])


def generate(m, prompt, n_steps, temperature=0.0, top_k=0, seed=0, eos_id=-1, max_seq=None):
    """Decode up to n_steps tokens; stops after emitting eos_id.  Returns
    (ids, logits [len(ids), V])."""
    kv = m.new_cache(max_seq or (len(prompt) + n_steps))
    tok, pos = llama.prefill(m, kv, prompt)
    ids, logits = [], []
    for _ in range(n_steps):
        lg = llama.decode_step(m, kv, tok, pos)
        tok = select(lg, temperature, top_k, pos, seed)
        ids.append(tok)
        logits.append(lg)
        pos += 1
        if tok == eos_id:
            break
    return np.array(ids, np.int32), np.stack(logits)
