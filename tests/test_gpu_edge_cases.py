"""The delta rule's own edge cases on the device, against the fp64 oracle (needs a GPU).

The oracle pins (tests/pins.py) fix these cases on the CPU; here the same constructions run
through every device path: the tensor-core prefill (bf16, dk = dv = 128), the SIMT prefill
(fp32, dk = dv = 64) and the decode kernel (one token per call). Each comparison prints a
"PARITY" line with its error and margin.

Cases (sources):
  * write-then-read: beta = 1 and an exactly unit key, so the read-out with q = k equals the
    value just written, whatever the decay and history (K3 explainer, section 2: the write
    predicts from memory and stores the error);
  * the explainer's four-message example, section 2 (tests/golden fixture), padded to the
    kernel width and repeated so one key is written 64 times inside every chunk: the read-out
    is always the latest status, never a sum;
  * alpha = 1 with orthonormal keys: a query with key j returns the last value written with
    key j (K3 training overview, section 2 "KDA": delta-rule corrective write);
  * beta = 0 from a non-zero initial state: no write, pure channel-wise decay of S0 (the same
    page: channel-wise forget gate);
  * half of every chunk re-writing one key with beta = 1, the rest random: the intra-chunk
    matrix strict_lower(diag(beta) K~ K^T) is as large as it gets, the hardest case for the
    chunked (I + M)^{-1}.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from linear_attention_05_gb300 import binding as B
from linear_attention_05_gb300 import inputs
from util import TOL, check, np32

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "delta_rule_project_status.txt")

# (name, dtype, d): the tensor-core path and the SIMT path
PATHS = [("tc", torch.bfloat16, 128), ("simt", torch.float32, 64)]


def _unit_keys(rng, n, d):
    """Keys with four entries of +-1/2 and the rest 0: exactly unit length in bf16 too."""
    keys = np.zeros((n, d), dtype=np.float32)
    for i in range(n):
        idx = rng.choice(d, 4, replace=False)
        keys[i, idx] = 0.5 * rng.choice([-1.0, 1.0], 4)
    return keys


def _block_hadamard(d):
    """d orthonormal keys with entries 0 and +-1/2: a 4 x 4 Hadamard block on each group of
    four channels (exact in bf16)."""
    h4 = 0.5 * np.array([[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]],
                        dtype=np.float32)
    keys = np.zeros((d, d), dtype=np.float32)
    for g in range(d // 4):
        keys[4 * g:4 * g + 4, 4 * g:4 * g + 4] = h4
    return keys


def _recipe(T, H, dk, dv, seed):
    """Recipe inputs (CPU fp32) as a starting point for the constructions."""
    x = inputs.tokens(T, H, dk, dv, torch.float32, seed=seed, device="cpu")
    return {n: t.numpy().copy() for n, t in x.items()}


def _dev(x, dtype):
    return {n: (None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV, dtype))
            for n, a in x.items()}


def _oracle(xd, cu, S0=None, l2norm=True, scale=1.0):
    g = None if xd["gate"] is None else np32(xd["gate"])
    s0 = None if S0 is None else np32(S0).astype(np.float64)
    return oracle.forward(np32(xd["q"]), np32(xd["k"]), np32(xd["v"]), np32(xd["log_alpha"]),
                          np32(xd["beta"]), g, s0, cu, scale=scale, l2norm=l2norm)


def _chunk(xd, cu, S0=None, l2norm=True, scale=1.0):
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    out, fs = B.chunk_fwd(xd["q"], xd["k"], xd["v"], xd["log_alpha"], xd["beta"], xd["gate"],
                          S0, cu_t, n_seq=len(cu) - 1, scale=scale, l2norm=l2norm)
    assert B.kda_get_error() == B.KDA_OK
    return out, fs


def _decode(xd, n_seq, T, S0, l2norm=True, scale=1.0):
    """Run T decode steps over n_seq equal-length sequences packed sequence-major
    ([n_seq * T] tokens); returns the outputs in the same packing and the final state."""
    H = xd["k"].shape[1]
    S = S0.clone().contiguous()
    out = torch.empty_like(xd["v"])

    def tok(name, t):
        a = xd[name]
        return None if a is None else a.view(n_seq, T, *a.shape[1:])[:, t].contiguous()

    for t in range(T):
        o = B.decode_step(tok("q", t), tok("k", t), tok("v", t), tok("log_alpha", t),
                          tok("beta", t), tok("gate", t), S, scale=scale, l2norm=l2norm)
        out.view(n_seq, T, H, -1)[:, t] = o
    assert B.kda_get_error() == B.KDA_OK
    return out, S


# ------------------------------------------------------------------------ write-then-read
def _write_then_read(dtype, d, n_seq=2, T=200, H=2, seed=400):
    x = _recipe(n_seq * T, H, d, d, seed)
    rng = np.random.default_rng(seed)
    for h in range(H):
        x["k"][:, h] = _unit_keys(rng, n_seq * T, d)
    x["q"] = x["k"].copy()
    x["beta"][:] = 1.0
    x["gate"] = None
    xd = _dev(x, dtype)
    return xd, [i * T for i in range(n_seq + 1)]


@pytest.mark.parametrize("path,dtype,d", PATHS)
def test_write_then_read_prefill(path, dtype, d):
    xd, cu = _write_then_read(dtype, d)
    S0 = inputs.state(len(cu) - 1, 2, d, d, seed=401, device=DEV)
    out, fs = _chunk(xd, cu, S0=S0, l2norm=False)
    ro, rs = _oracle(xd, cu, S0=S0, l2norm=False)
    check(f"write_then_read/{path}/out_vs_oracle", np32(out), ro, TOL[dtype])
    check(f"write_then_read/{path}/state_vs_oracle", np32(fs), rs, TOL[dtype])
    # the read-out is the value just written (exact in the mathematics)
    check(f"write_then_read/{path}/out_vs_v", np32(out), np32(xd["v"]), TOL[dtype])


def test_write_then_read_decode():
    T, n_seq = 100, 3
    xd, cu = _write_then_read(torch.bfloat16, 128, n_seq=n_seq, T=T)
    S0 = inputs.state(n_seq, 2, 128, 128, seed=402, device=DEV)
    out, S = _decode(xd, n_seq, T, S0, l2norm=False)
    ro, rs = _oracle(xd, cu, S0=S0, l2norm=False)
    check("write_then_read/decode/out_vs_oracle", np32(out), ro, TOL[torch.bfloat16])
    check("write_then_read/decode/state_vs_oracle", np32(S), rs, TOL[torch.bfloat16])
    check("write_then_read/decode/out_vs_v", np32(out), np32(xd["v"]), TOL[torch.bfloat16])


# ------------------------------------------------------------------------ four messages
def _golden():
    fx = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                name, *vals = line.split()
                fx.setdefault(name, []).append([float(v) for v in vals])
    return fx


def _four_messages(dtype, d, T=256, H=2):
    """The fixture's key (dk 4) and one-hot status codes (dv 4), zero-padded to d channels.
    Token t writes status t % 4 (development, delayed, approved, completed, again), so every
    64-token chunk writes the same key 64 times; beta = 1, no forgetting, q = k."""
    fx = _golden()
    key = np.zeros(d, np.float32)
    key[:len(fx["key"][0])] = fx["key"][0]
    codes = np.zeros((4, d), np.float32)
    codes[:, :4] = np.array(fx["value"], np.float32)
    expect = np.zeros((4, d), np.float32)
    expect[:, :4] = np.array(fx["expect"], np.float32)
    st = np.arange(T) % 4
    k = np.broadcast_to(key, (T, H, d)).copy()
    x = {"q": k.copy(), "k": k, "v": np.broadcast_to(codes[st][:, None, :], (T, H, d)).copy(),
         "beta": np.ones((T, H), np.float32), "log_alpha": np.zeros((T, H, d), np.float32),
         "gate": None}
    want = np.broadcast_to(expect[st][:, None, :], (T, H, d))
    return _dev(x, dtype), [0, T], want


@pytest.mark.parametrize("path,dtype,d", PATHS)
def test_four_messages_prefill(path, dtype, d):
    xd, cu, want = _four_messages(dtype, d)
    out, fs = _chunk(xd, cu, l2norm=False)
    ro, rs = _oracle(xd, cu, l2norm=False)
    assert np.array_equal(ro, want)  # the oracle reads the latest status, exactly
    check(f"four_messages/{path}/out_vs_expected", np32(out), want, TOL[dtype])
    check(f"four_messages/{path}/state_vs_oracle", np32(fs), rs, TOL[dtype])
    # with the library's L2 normalisation the key is k / sqrt(1 + 1e-6): still the latest code
    out2, fs2 = _chunk(xd, cu, l2norm=True)
    ro2, rs2 = _oracle(xd, cu, l2norm=True)
    check(f"four_messages/{path}/l2norm_out_vs_oracle", np32(out2), ro2, TOL[dtype])
    check(f"four_messages/{path}/l2norm_state_vs_oracle", np32(fs2), rs2, TOL[dtype])


def test_four_messages_decode():
    xd, cu, want = _four_messages(torch.bfloat16, 128, T=96)
    S0 = torch.zeros((1, 2, 128, 128), dtype=torch.float32, device=DEV)
    out, S = _decode(xd, 1, 96, S0, l2norm=False)
    _, rs = _oracle(xd, cu, l2norm=False)
    check("four_messages/decode/out_vs_expected", np32(out), want, TOL[torch.bfloat16])
    check("four_messages/decode/state_vs_oracle", np32(S), rs, TOL[torch.bfloat16])


# ------------------------------------------------------------------------ orthonormal retrieval
def _retrieval(dtype, d, T=300, H=2, seed=410):
    """alpha = 1, beta = 1; token t writes v_t with key w_t and queries key r_t (both drawn
    from d orthonormal keys, the writes from half of them so that keys repeat inside a
    chunk)."""
    rng = np.random.default_rng(seed)
    basis = _block_hadamard(d)
    x = _recipe(T, H, d, d, seed)
    for h in range(H):
        w = rng.integers(0, d // 2, T)
        r = np.where(rng.random(T) < 0.8, w[rng.integers(0, T, T)], rng.integers(0, d, T))
        x["k"][:, h] = basis[w]
        x["q"][:, h] = basis[r]
    x["beta"][:] = 1.0
    x["log_alpha"][:] = 0.0
    x["gate"] = None
    return _dev(x, dtype), [0, T]


def _retrieval_expected(xd):
    """The read-out the definition gives: the last value written with the query's key up to
    and including token t (zero if none), built from the values the device sees."""
    v = np32(xd["v"]).astype(np.float64)
    k = np32(xd["k"])
    q = np32(xd["q"])
    T, H, d = v.shape
    out = np.zeros((T, H, d))
    for h in range(H):
        last = {}
        for t in range(T):
            last[k[t, h].tobytes()] = v[t, h]
            out[t, h] = last.get(q[t, h].tobytes(), np.zeros(d))
    return out


@pytest.mark.parametrize("path,dtype,d", PATHS)
def test_orthonormal_retrieval_prefill(path, dtype, d):
    xd, cu = _retrieval(dtype, d)
    want = _retrieval_expected(xd)
    out, fs = _chunk(xd, cu, l2norm=False)
    ro, rs = _oracle(xd, cu, l2norm=False)
    assert np.max(np.abs(ro - want)) < 1e-12  # the oracle retrieves exactly
    check(f"orthonormal/{path}/out_vs_expected", np32(out), want, TOL[dtype])
    check(f"orthonormal/{path}/state_vs_oracle", np32(fs), rs, TOL[dtype])


def test_orthonormal_retrieval_decode():
    T = 120
    xd, cu = _retrieval(torch.bfloat16, 128, T=T)
    want = _retrieval_expected(xd)
    S0 = torch.zeros((1, 2, 128, 128), dtype=torch.float32, device=DEV)
    out, S = _decode(xd, 1, T, S0, l2norm=False)
    _, rs = _oracle(xd, cu, l2norm=False)
    check("orthonormal/decode/out_vs_expected", np32(out), want, TOL[torch.bfloat16])
    check("orthonormal/decode/state_vs_oracle", np32(S), rs, TOL[torch.bfloat16])


# ------------------------------------------------------------------------ beta = 0
@pytest.mark.parametrize("path,dtype,d", PATHS)
def test_beta_zero_pure_decay_prefill(path, dtype, d):
    lengths = [130, 64, 1, 200]
    cu = [0] + np.cumsum(lengths).tolist()
    x = _recipe(cu[-1], 3, d, d, 420)
    x["beta"][:] = 0.0
    xd = _dev(x, dtype)
    S0 = inputs.state(len(lengths), 3, d, d, seed=421, device=DEV)
    out, fs = _chunk(xd, cu, S0=S0, scale=0.9)
    ro, rs = _oracle(xd, cu, S0=S0, scale=0.9)
    check(f"beta_zero/{path}/out_vs_oracle", np32(out), ro, TOL[dtype])
    check(f"beta_zero/{path}/state_vs_oracle", np32(fs), rs, TOL[dtype])
    # closed form of the final state: Diag(exp(sum log_alpha)) S0
    la = np32(xd["log_alpha"]).astype(np.float64)
    s0 = np32(S0).astype(np.float64)
    for s in range(len(lengths)):
        G = la[cu[s]:cu[s + 1]].sum(0)  # [H, d]
        check(f"beta_zero/{path}/closed_form_state_seq{s}", np32(fs[s]),
              np.exp(G)[:, :, None] * s0[s], TOL[dtype])


def test_beta_zero_decode():
    T, n_seq, d = 70, 2, 128
    x = _recipe(n_seq * T, 2, d, d, 422)
    x["beta"][:] = 0.0
    xd = _dev(x, torch.bfloat16)
    S0 = inputs.state(n_seq, 2, d, d, seed=423, device=DEV)
    out, S = _decode(xd, n_seq, T, S0)
    ro, rs = _oracle(xd, [0, T, 2 * T], S0=S0)
    check("beta_zero/decode/out_vs_oracle", np32(out), ro, TOL[torch.bfloat16])
    check("beta_zero/decode/state_vs_oracle", np32(S), rs, TOL[torch.bfloat16])


# ------------------------------------------------------------------------ repeated key, beta ~ 1
def _repeated_key(dtype, d, lengths, H=2, seed=430):
    """In every chunk the even tokens write one fixed unit key with beta = 1, the odd tokens
    random keys with recipe beta."""
    cu = [0] + np.cumsum(lengths).tolist()
    x = _recipe(cu[-1], H, d, d, seed)
    rng = np.random.default_rng(seed)
    star = _unit_keys(rng, H, d)
    pos = np.arange(cu[-1])
    even = (pos % 2) == 0
    for h in range(H):
        x["k"][even, h] = star[h]
    x["beta"][even] = 1.0
    return _dev(x, dtype), cu


@pytest.mark.parametrize("path,dtype,d", PATHS)
def test_repeated_key_half_chunk_prefill(path, dtype, d):
    xd, cu = _repeated_key(dtype, d, [256, 191, 65])
    S0 = inputs.state(3, 2, d, d, seed=431, device=DEV)
    out, fs = _chunk(xd, cu, S0=S0)
    ro, rs = _oracle(xd, cu, S0=S0)
    check(f"repeated_key/{path}/out_vs_oracle", np32(out), ro, TOL[dtype])
    check(f"repeated_key/{path}/state_vs_oracle", np32(fs), rs, TOL[dtype])


def test_repeated_key_all_tokens_alpha_one():
    """One key written by every token with beta = 1 and no forgetting over 8 chunks: the
    intra-chunk matrix is the all-ones strict lower triangle."""
    T, d = 512, 128
    x = _recipe(T, 2, d, d, 440)
    star = _unit_keys(np.random.default_rng(440), 2, d)
    x["k"][:] = star[None]
    x["beta"][:] = 1.0
    x["log_alpha"][:] = 0.0
    xd = _dev(x, torch.bfloat16)
    S0 = inputs.state(1, 2, d, d, seed=441, device=DEV)
    out, fs = _chunk(xd, [0, T], S0=S0, l2norm=False)
    ro, rs = _oracle(xd, [0, T], S0=S0, l2norm=False)
    check("repeated_key_all/tc/out_vs_oracle", np32(out), ro, TOL[torch.bfloat16])
    check("repeated_key_all/tc/state_vs_oracle", np32(fs), rs, TOL[torch.bfloat16])


def test_repeated_key_decode():
    T, n_seq, d = 90, 2, 128
    xd, cu = _repeated_key(torch.bfloat16, d, [T] * n_seq)
    S0 = inputs.state(n_seq, 2, d, d, seed=432, device=DEV)
    out, S = _decode(xd, n_seq, T, S0)
    ro, rs = _oracle(xd, cu, S0=S0)
    check("repeated_key/decode/out_vs_oracle", np32(out), ro, TOL[torch.bfloat16])
    check("repeated_key/decode/state_vs_oracle", np32(S), rs, TOL[torch.bfloat16])
