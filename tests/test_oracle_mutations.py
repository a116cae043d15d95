"""Plant one plausible mistake at a time in a private copy of the CPU oracle and check that the
pins catch it.  Nothing here touches a GPU; the mistakes live only in the in-memory copy."""
import os
import types

import pytest

import oracle_pins as pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "qspec_oracle.py")

# (name, text in the oracle, replacement)
MUTATIONS = [
    ("bf16 ties away from zero", "r = np.rint(xf / spacing) * spacing",
     "r = np.trunc(xf / spacing + np.copysign(0.5, xf)) * spacing"),
    ("bf16 rounded through fp32 first", "x = np.asarray(x, dtype=np.float64)\n    out = np.array(x, copy=True)",
     "x = np.asarray(x, dtype=np.float32).astype(np.float64)\n    out = np.array(x, copy=True)"),
    ("bf16 subnormal exponent floor off by one", "e = np.maximum(e2 - 1, -126)", "e = np.maximum(e2 - 1, -127)"),
    ("bf16 overflows at the largest finite value", "r = np.where(np.abs(r) > bf16_max,",
     "r = np.where(np.abs(r) >= bf16_max,"),
    ("weight divisor 8", "s32 = amax / np.float32(7.0)", "s32 = amax / np.float32(8.0)"),
    ("weight scale not fp16-rounded before coding", "s = S.astype(np.float32)[:, :, None]",
     "s = s32[:, :, None]"),
    ("weight rounding half up", "q = np.clip(np.rint(q), -8, 7)", "q = np.clip(np.floor(q + 0.5), -8, 7)"),
    ("nibble order swapped", "byte = nib[:, :, 0::2] | (nib[:, :, 1::2] << 4)", "byte = nib[:, :, 1::2] | (nib[:, :, 0::2] << 4)"),
    ("natural channel order in a word", "WORD_ORDER = (0, 2, 4, 6, 1, 3, 5, 7)", "WORD_ORDER = (0, 1, 2, 3, 4, 5, 6, 7)"),
    ("unpack without sign", "out = np.where(out >= 8, out - 16, out)", "out = out"),
    ("group scale tiled instead of repeated", "scale = np.repeat(S.astype(np.float64), GROUP, axis=1)",
     "scale = np.tile(S.astype(np.float64), (1, GROUP))"),
    ("w4a16 transposed operand", "return x @ Wd.T", "return (Wd @ x.T)"),
    ("activation divisor a power of two", "qmax = 2 ** (bits - 1) - 1", "qmax = 2 ** (bits - 1)"),
    ("activation scale rounded to fp16", "s_a = (amax / np.float32(qmax)).astype(np.float32)",
     "s_a = (amax / np.float32(qmax)).astype(np.float16).astype(np.float32)"),
    ("activation codes clamped asymmetrically", "np.clip(np.rint(x[m] / s_a[m]), -qmax - 1, qmax)",
     "np.clip(np.rint(x[m] / s_a[m]), -qmax, qmax - 1)"),
    ("W4A8 quantises to 4 bits", "return linear_w4a4(x_bits, Wp, S, rows, bits=8)",
     "return linear_w4a4(x_bits, Wp, S, rows, bits=4)"),
    ("w4a4 drops the token scale", "y = s_a.astype(np.float64)[:, None] * np.einsum",
     "y = 1.0 * np.einsum"),
    ("w4a4 groups strided", 'acc = np.einsum("mgk,ngk->mng", qa.reshape(M, G, GROUP), codes.reshape(N, G, GROUP))',
     'acc = np.einsum("mkg,nkg->mng", qa.reshape(M, GROUP, G), codes.reshape(N, GROUP, G))'),
    ("softmax without max shift", "e = np.exp(l - m)", "e = np.exp(l)"),
    ("argmax takes the last tie", "return int(hits[0])", "return int(hits[-1])"),
    ("greedy drops the target token", "out[b, k] = t[b, k]", "out[b, k] = t[b, k] if k < gamma else -1"),
    ("greedy compares with the next position", "int(d[b, k]) == int(t[b, k])", "int(d[b, k]) == int(t[b, k + 1])"),
    ("accept test not strict", "if not (float(u_acc[i]) < a[i]):", "if not (float(u_acc[i]) <= a[i]):"),
    ("residual keeps negative mass", "r = np.maximum(0.0, p_rows[n] - q_rows[n])", "r = np.abs(p_rows[n] - q_rows[n])"),
    ("rejection resamples from p", "r = np.maximum(0.0, p_rows[n] - q_rows[n])", "r = p_rows[n]"),
    ("bonus drawn from the last draft row", "r = p_rows[gamma]", "r = q_rows[gamma - 1]"),
    ("acceptance ratio inverted", "min(1.0, p_tok[i] / q_tok[i])", "min(1.0, q_tok[i] / p_tok[i])"),
    ("resample uniform not indexed by n", "j = inverse_cdf(r, float(u_res[n]))", "j = inverse_cdf(r, float(u_res[0]))"),
    ("inverse cdf non-strict", "hit = np.nonzero(c > u * R)[0]", "hit = np.nonzero(c >= u * R)[0]"),
    ("top-1 probability of the draft taken at the target's token", "d_p[b, i] = softmax(Ld[b, i])[d_tok[b, i]]",
     "d_p[b, i] = softmax(Ld[b, i])[t_tok[b, i]]"),
    ("high-confidence test not strict", "if t_p[b, i] > high and d_p[b, i] > high:",
     "if t_p[b, i] >= high and d_p[b, i] >= high:"),
    ("low region counts either mode at or below", "if t_p[b, i] <= high and d_p[b, i] <= high:",
     "if t_p[b, i] <= high or d_p[b, i] <= high:"),
    ("decode loop drops the token after the accepted drafts", "seq += [int(t) for t in out[:n + 1]]",
     "seq += [int(t) for t in out[:n]]"),
    ("target scores each position one token late", "tl = np.stack([target(seq + d[:i]) for i in range(gamma + 1)])[None]",
     "tl = np.stack([target(seq + d[:i + 1]) for i in range(gamma + 1)])[None]"),
    ("draft does not see its own tokens", "l = draft(seq + d)", "l = draft(seq)"),
    ("toy model runs verify mode when drafting", 'y = linear_w4a4(x, Wp, S)["y"] if draft_mode else linear_w4a16(x, Wp, S)',
     "y = linear_w4a16(x, Wp, S)"),
    ("tree walk scores a child with its own row", "children = [j for j in range(T) if valid[j] and int(par[b, j]) == cur and int(tok[b, j]) == t[row]]",
     "children = [j for j in range(T) if valid[j] and int(par[b, j]) == cur and int(tok[b, j]) == t[j + 1]]"),
    ("tree walk takes the highest-index sibling", "cur = min(children)", "cur = max(children)"),
    ("tree walk ignores the parent", "children = [j for j in range(T) if valid[j] and int(par[b, j]) == cur and int(tok[b, j]) == t[row]]",
     "children = [j for j in range(T) if valid[j] and j > cur and int(tok[b, j]) == t[row]]"),
    ("E[T] exponent off by one", "return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)",
     "return (1.0 - alpha ** gamma) / (1.0 - alpha)"),
]


def mutated_oracle(old, new):
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


def caught(mod):
    checks = list(pins.ALL_FAST) + [pins.check_sampling_exact_marginal,
                                    lambda o: pins.check_expected_tokens(o, trials=40_000)]
    for check in checks:
        try:
            check(mod)
        except Exception:
            return True
    return False


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new):
    assert caught(mutated_oracle(old, new)), f"no pin catches: {name}"


def test_unmutated_copy_passes():
    src = open(SRC, encoding="utf-8").read()
    mod = types.ModuleType("oracle_copy")
    exec(compile(src, "oracle_copy", "exec"), mod.__dict__)
    for check in pins.ALL_FAST:
        check(mod)
