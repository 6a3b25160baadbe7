"""Plain fp64 attention definitions (test infrastructure, see package docstring).

Sources, by page and section:

* "MiniCPM4 `forward_step` Attention Performance Fix", section 4.1 (the
  replacement ``forward_step``): the new key/value rows are written into the
  static cache at ``position_id`` *before* attention, then the query attends
  the cache slice ``[:position_id + 1]`` with ``enable_gqa=True``.  Section 3
  states that this slice alone enforces causality (no mask) and that at
  position 0 the softmax over a single entry is the identity.
* Same page, section 2.1/2.3 (the original code): a full-length boolean mask
  ``arange(max_len) <= position_id`` over the whole cache.  It gives the same
  result; it is kept here only as ``decode_masked_full`` so tests can check
  the equivalence.
* "step14_3 -- batched attention", section "problem" (per-head loop): for one
  head, scores = q_h k_h^T / sqrt(d_head), masked positions set to -inf,
  softmax over keys, weights times v_h.  The scale is an explicit argument
  here; the decode page calls SDPA without ``scale``, whose default is
  1/sqrt(D).
* Same page, section "F.scaled_dot_product_attention": prefill of new tokens
  over ``K_full``/``V_full`` that include the cached prefix.  New token i (at
  absolute position start_pos + i) attends keys 0..start_pos + i (the causal
  mask aligned to the bottom-right corner).

GQA head mapping: query head h reads KV head floor(h / g), g = Hq / Hkv (the
repeat-KV convention of PyTorch's ``enable_gqa``).

All arithmetic is float64 on the exact values of the (bf16) inputs.
"""

from __future__ import annotations

import numpy as np


# --- small named steps (kept separate so tests can plant mistakes in them) ---

def _kv_head(h: int, g: int, Hkv: int) -> int:
    """KV head read by query head h: contiguous groups of g query heads."""
    return h // g


def _attended_rows(position: int) -> range:
    """Cache rows a decode step at ``position`` attends: 0..position inclusive."""
    return range(0, position + 1)


def _causal_keys(start_pos: int, i: int) -> range:
    """Keys visible to new token i of a prefill over a start_pos-long prefix."""
    return range(0, start_pos + i + 1)


def _softmax(s: np.ndarray) -> np.ndarray:
    """Softmax over the last axis (max-subtracted; mathematically exact)."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def _attend(q_h: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """One query row over keys K [n, D] and values V [n, D]."""
    s = scale * (K @ q_h)          # [n] scores
    w = _softmax(s)                # [n] weights
    return w @ V                   # [D]


# --- public definitions ------------------------------------------------------

def kv_append(k_cache, v_cache, k_new, v_new, positions):
    """In-place row write of the decode page, section 4.1:
    ``key_cache[:, :, position_id, :] = key_states`` (same for values),
    one ``position_id`` per sequence.  Returns new arrays; the inputs are not
    modified.  Works for any dtype (the tests compare bf16 bit patterns)."""
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    B, Hkv = kc.shape[0], kc.shape[1]
    for b in range(B):
        p = int(positions[b])
        for h in range(Hkv):
            kc[b, h, p, :] = k_new[b, h, :]
            vc[b, h, p, :] = v_new[b, h, :]
    return kc, vc


def decode_rows(q, k_cache, v_cache, positions, scale, rows):
    """Decode output for selected (b, h) rows only: returns [len(rows), D].

    ``k_cache``/``v_cache`` must already contain this step's appended row.
    """
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    g = Hq // Hkv
    out = np.empty((len(rows), D), dtype=np.float64)
    for r, (b, h) in enumerate(rows):
        kvh = _kv_head(h, g, Hkv)
        idx = list(_attended_rows(int(positions[b])))
        K = np.asarray(k_cache[b, kvh, idx, :], dtype=np.float64)
        V = np.asarray(v_cache[b, kvh, idx, :], dtype=np.float64)
        out[r] = _attend(np.asarray(q[b, h], dtype=np.float64), K, V, scale)
    return out


def decode(q, k_cache, v_cache, positions, scale):
    """Sliced decode attention of the decode page, section 3/4.1.

    q [B, Hq, D]; k_cache, v_cache [B, Hkv, L, D] (after this step's append);
    positions [B].  Returns out [B, Hq, D] float64.
    """
    B, Hq, D = q.shape
    rows = [(b, h) for b in range(B) for h in range(Hq)]
    return decode_rows(q, k_cache, v_cache, positions, scale, rows).reshape(B, Hq, D)


def decode_masked_full(q, k_cache, v_cache, positions, scale):
    """The original decode of the decode page, section 2.1/2.3: attend all L
    cache rows with the boolean mask ``arange(L) <= position_id`` (masked
    scores are -inf, so their weight is exactly zero).  Same result as
    ``decode``; present only so tests can check that equivalence."""
    B, Hq, D = q.shape
    Hkv, L = k_cache.shape[1], k_cache.shape[2]
    g = Hq // Hkv
    out = np.empty((B, Hq, D), dtype=np.float64)
    for b in range(B):
        mask = np.arange(L) <= int(positions[b])
        for h in range(Hq):
            kvh = _kv_head(h, g, Hkv)
            K = np.asarray(k_cache[b, kvh], dtype=np.float64)
            V = np.asarray(v_cache[b, kvh], dtype=np.float64)
            s = scale * (K @ np.asarray(q[b, h], dtype=np.float64))
            s = np.where(mask, s, -np.inf)
            w = _softmax(s)
            # rows outside the mask carry weight 0; keep NaN/inf there out
            out[b, h] = w[mask] @ V[mask]
    return out


def prefill_rows(q, k, v, start_pos, scale, rows):
    """Prefill output for selected (i, h) rows: returns [len(rows), d]."""
    S, Hq, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    out = np.empty((len(rows), d), dtype=np.float64)
    for r, (i, h) in enumerate(rows):
        kvh = _kv_head(h, g, Hkv)
        idx = list(_causal_keys(int(start_pos), int(i)))
        K = np.asarray(k[idx, kvh, :], dtype=np.float64)
        V = np.asarray(v[idx, kvh, :], dtype=np.float64)
        out[r] = _attend(np.asarray(q[i, h], dtype=np.float64), K, V, scale)
    return out


def prefill(q, k, v, start_pos, scale):
    """Causal prefill over a cached prefix (prefill page, SDPA section; decode
    page section 5: batch prefill is causal).

    q [S, Hq, d] new tokens at absolute positions start_pos..start_pos+S-1;
    k, v [start_pos + S, Hkv, d] prefix rows first.  Returns [S, Hq, d].
    """
    S, Hq, d = q.shape
    rows = [(i, h) for i in range(S) for h in range(Hq)]
    return prefill_rows(q, k, v, start_pos, scale, rows).reshape(S, Hq, d)


# --- local-window decode -----------------------------------------------------
#
# Attend only the most recent W cache rows.  The reading taken: rows
# max(0, pos - W + 1) .. pos inclusive (W keys, the current one included);
# W >= pos + 1 is the full decode above.

def _window_rows(position: int, window: int) -> range:
    """Cache rows a windowed decode step at ``position`` attends."""
    return range(max(0, position - window + 1), position + 1)


def decode_window(q, k_cache, v_cache, positions, scale, window):
    """Decode over the last ``window`` rows up to each sequence's position.

    q [B, Hq, D]; caches [B, Hkv, L, D] (after this step's append).  Returns
    out [B, Hq, D] float64."""
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    g = Hq // Hkv
    out = np.empty((B, Hq, D), dtype=np.float64)
    for b in range(B):
        idx = list(_window_rows(int(positions[b]), int(window)))
        for h in range(Hq):
            kvh = _kv_head(h, g, Hkv)
            K = np.asarray(k_cache[b, kvh, idx, :], dtype=np.float64)
            V = np.asarray(v_cache[b, kvh, idx, :], dtype=np.float64)
            out[b, h] = _attend(np.asarray(q[b, h], dtype=np.float64), K, V, scale)
    return out


# --- multi-token decode --------------------------------------------------------
#
# S new tokens per sequence (e.g. draft tokens to verify): token t of
# sequence b sits at position positions[b] + t and attends cache rows
# 0 .. positions[b] + t (its own row included, later new tokens not).  The
# cache already holds the S new rows.

def decode_multi(q, k_cache, v_cache, positions, scale):
    """q [B, S, Hq, D]; caches [B, Hkv, L, D] holding rows up to
    positions[b] + S - 1.  Returns out [B, S, Hq, D] float64."""
    B, S, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    g = Hq // Hkv
    out = np.empty((B, S, Hq, D), dtype=np.float64)
    for b in range(B):
        for t in range(S):
            idx = list(_attended_rows(int(positions[b]) + t))
            for h in range(Hq):
                kvh = _kv_head(h, g, Hkv)
                K = np.asarray(k_cache[b, kvh, idx, :], dtype=np.float64)
                V = np.asarray(v_cache[b, kvh, idx, :], dtype=np.float64)
                out[b, t, h] = _attend(np.asarray(q[b, t, h], dtype=np.float64), K, V, scale)
    return out


# --- rotary position embedding (decode page, section 4.1) --------------------
#
# The decode page rotates q and the new k with apply_rotary_pos_emb(q, k,
# cos, sin) before the cache write, without defining it.  The reading taken
# is the rotate-half form: x' = x * cos + rotate_half(x) * sin with
# rotate_half(x) = [-x[D/2:], x[:D/2]], computed in fp32 one IEEE operation
# at a time (product, product, sum; no fused multiply-add), with the rotated
# key rounded to bf16 (round to nearest even) for the bf16 cache and the
# rotated query kept in fp32.

def rope_f32(x, cos, sin):
    """x [..., D] (bf16 values), cos/sin [..., D] fp32 -> fp32 rotated x."""
    x = np.asarray(x, dtype=np.float32)
    c = np.asarray(cos, dtype=np.float32)
    s = np.asarray(sin, dtype=np.float32)
    half = x.shape[-1] // 2
    rot = np.concatenate([-x[..., half:], x[..., :half]], axis=-1)
    return (x * c) + (rot * s)          # float32 ops, each rounded


def round_bf16(x):
    """fp32 -> nearest bf16 value (ties to even), returned as float64."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def decode_rope_step(q, k_new, v_new, cos, sin, k_cache, v_cache, positions, scale):
    """One decode step with rotary embedding: rotate q and the new k at each
    sequence's position, append (rotated k as bf16, v as is), attend.

    q [B,Hq,D]; k_new, v_new [B,Hkv,D]; cos, sin [B,D] (the rotation at
    positions[b], shared by all heads); caches [B,Hkv,L,D].  Returns
    (out [B,Hq,D] float64, k_cache, v_cache after the append)."""
    B = q.shape[0]
    q_rot = rope_f32(q, np.asarray(cos)[:, None, :], np.asarray(sin)[:, None, :])
    k_rot = round_bf16(rope_f32(k_new, np.asarray(cos)[:, None, :], np.asarray(sin)[:, None, :]))
    kc, vc = kv_append(k_cache, v_cache, k_rot, v_new, positions)
    out = decode(q_rot.astype(np.float64), kc, vc, positions, scale)
    assert out.shape[0] == B
    return out, kc, vc


# --- algorithmic work (the counts the roofline divides by) -------------------

def decode_bytes(positions, Hq, Hkv, D, elem=2):
    """Bytes a decode step must move: K and V rows 0..pos_b of every KV head,
    plus q in and out.  The full-length work the sliced method avoids is not
    counted."""
    n = sum(int(p) + 1 for p in positions)
    B = len(positions)
    return 2 * Hkv * n * D * elem + 2 * B * Hq * D * elem


def decode_flops(positions, Hq, D):
    """2*D flops for q.k plus 2*D for p*v, per (query head, attended row)."""
    n = sum(int(p) + 1 for p in positions)
    return 4 * D * Hq * n


def prefill_flops(S, start_pos, H, d):
    """QK^T and PV flops restricted to the causal keys: 4*d per (head, visible
    key) pair."""
    n = sum(start_pos + i + 1 for i in range(S))
    return 4 * d * H * n
