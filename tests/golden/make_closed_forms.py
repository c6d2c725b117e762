"""Write closed_forms.json: hand-derived cases of the decode-step attention block.

The pages print no worked numerical example, so these fixtures pin the oracle to
the mathematics instead: each case is small enough to solve by hand, and its
expected values are written here as the closed-form expressions of that
derivation, evaluated with the ``math`` module only (neither the oracle nor the
CUDA path is called). Run: ``python tests/golden/make_closed_forms.py``.
"""
import json
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def cases():
    out = []
    # RMSNorm with fused residual add (fusedtok README, "Operators": RMSNorm (+residual);
    # cutileGPT README, "Why tiles": rstd = 1/sqrt(sum(x*x)/N + eps)).
    # s = x + r = [3, 4]; mean(s^2) = 12.5; eps = 0.5 -> rstd = 1/sqrt(13).
    out.append({
        "name": "rmsnorm_residual_3_4",
        "source": "fusedtok README, Operators (RMSNorm (+residual)); cutileGPT README, Why tiles",
        "derivation": "s=[3,4], mean(s^2)=12.5, eps=0.5, rstd=1/sqrt(13), y=s*rstd*w",
        "x": [[1.0, 3.0]], "residual": [[2.0, 1.0]], "w": [2.0, 0.5], "eps": 0.5,
        "expect_y": [[6.0 / math.sqrt(13.0), 2.0 / math.sqrt(13.0)]],
        "expect_residual": [[3.0, 4.0]],
    })
    # RoPE, D = 4, theta = 1e4 -> inv_freq = [1, 1e4^(-1/2)] = [1, 0.01]; pos = 100 ->
    # angles [100, 1] rad (fusedtok README, Operators: RoPE interleaved and NeoX layouts).
    c100, s100, c1, s1 = math.cos(100.0), math.sin(100.0), math.cos(1.0), math.sin(1.0)
    out.append({
        "name": "rope_neox_d4",
        "source": "fusedtok README, Operators (RoPE, NeoX layout) and Usage (rope(..., neox=True))",
        "derivation": "NeoX pairs (0,2),(1,3); angles 100 and 1 rad",
        "x": [1.0, 2.0, 3.0, 4.0], "pos": 100, "theta": 1e4, "layout": "neox",
        "expect": [1 * c100 - 3 * s100, 2 * c1 - 4 * s1, 1 * s100 + 3 * c100, 2 * s1 + 4 * c1],
    })
    out.append({
        "name": "rope_interleaved_d4",
        "source": "fusedtok README, Operators (RoPE, interleaved layout)",
        "derivation": "interleaved pairs (0,1),(2,3); angles 100 and 1 rad",
        "x": [1.0, 2.0, 3.0, 4.0], "pos": 100, "theta": 1e4, "layout": "interleaved",
        "expect": [1 * c100 - 2 * s100, 1 * s100 + 2 * c100, 3 * c1 - 4 * s1, 3 * s1 + 4 * c1],
    })
    # QK-norm + RoPE + append (cutileGPT README, "The current runtime includes").
    # D=4, theta=9 -> inv_freq=[1, 1/3]; pos=3 -> angles [3, 1].
    # q=[3,4,0,0], w=1, eps=0 -> rms=2.5 -> [1.2,1.6,0,0]; NeoX pairs (0,2),(1,3).
    # k=[0,0,0,2], w=[1,1,1,2] -> rms=1 -> [0,0,0,4]; pair (1,3)=(0,4) rotates by 1 rad.
    c3, s3 = math.cos(3.0), math.sin(3.0)
    kc = [[[[0.5 * (t + 1) + 0.25 * d for d in range(4)] for t in range(5)]]]
    vc = [[[[-0.5 * (t + 1) + 0.125 * d for d in range(4)] for t in range(5)]]]
    kc_exp = json.loads(json.dumps(kc))
    vc_exp = json.loads(json.dumps(vc))
    kc_exp[0][0][3] = [0.0, -4.0 * s1, 0.0, 4.0 * c1]
    vc_exp[0][0][3] = [5.0, 6.0, 7.0, 8.0]
    out.append({
        "name": "qknorm_rope_append_d4",
        "source": "cutileGPT README, The current runtime includes (fused QK-Norm + RoPE + KV-cache writes)",
        "derivation": "see comments in make_closed_forms.py",
        "q": [[[3.0, 4.0, 0.0, 0.0]]], "k_new": [[[0.0, 0.0, 0.0, 2.0]]],
        "v_new": [[[5.0, 6.0, 7.0, 8.0]]], "q_norm_w": [1.0, 1.0, 1.0, 1.0],
        "k_norm_w": [1.0, 1.0, 1.0, 2.0], "eps": 0.0, "theta": 9.0, "layout": "neox",
        "pos": [3], "k_cache": kc, "v_cache": vc,
        "expect_q": [[[1.2 * c3, 1.6 * c1, 1.2 * s3, 1.6 * s1]]],
        "expect_k_cache": kc_exp, "expect_v_cache": vc_exp,
    })
    # GQA decode attention (fusedtok README, Operators: attention_decode).
    # D=2, Hq=2, Hkv=1, scale=1/sqrt(2). Head 0: q=[sqrt(2) ln 3, 0], keys [1,0],[0,0]
    # -> logits [ln 3, 0] -> weights [3/4, 1/4] -> out = 3/4 [4,0] + 1/4 [0,8] = [3,2].
    # Head 1: q=0 -> uniform weights -> mean of V = [2,4]. Slot 2 is past len and holds NaN.
    nan = float("nan")
    out.append({
        "name": "attention_two_keys",
        "source": "fusedtok README, Operators (attention_decode) and Benchmarks (repeat_interleave heads)",
        "derivation": "logits [ln3, 0] -> softmax [3/4, 1/4]; q=0 -> mean of V",
        "q": [[[math.sqrt(2.0) * math.log(3.0), 0.0], [0.0, 0.0]]],
        "k_cache": [[[[1.0, 0.0], [0.0, 0.0], [nan, nan]]]],
        "v_cache": [[[[4.0, 0.0], [0.0, 8.0], [nan, nan]]]],
        "lens": [2],
        "expect": [[[3.0, 2.0], [2.0, 4.0]]],
    })
    # Split merge: chunk A o=[1,0], lse=0; chunk B o=[0,1], lse=ln 3 -> weights 1/4, 3/4.
    out.append({
        "name": "merge_two_chunks",
        "source": "fusedtok README, Operators (flash-decoding split over long caches)",
        "derivation": "weights e^0 : e^ln3 = 1 : 3",
        "o": [[1.0, 0.0], [0.0, 1.0]], "lse": [0.0, math.log(3.0)],
        "expect": [0.25, 0.75],
    })
    return out


def main():
    path = os.path.join(HERE, "closed_forms.json")
    with open(path, "w") as f:
        json.dump(cases(), f, indent=1, allow_nan=True)
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
