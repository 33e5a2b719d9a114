"""Writes handworked.json: closed-form attention results derived by hand.

The pages print no numeric worked example, so these cases are derived from the
definition of softmax attention (scores, stable softmax, weighted sum, row
logsumexp, softmax-Jacobian backward) with inputs chosen so every quantity is
a closed form.  No oracle or GPU code is called: the numbers below are the
derivations evaluated with ``math``.

Run from the repository root:  python tests/golden/make_handworked.py
"""
import json
import math
import os

LN3, LN9 = math.log(3.0), math.log(9.0)

CASES = {
    "source": "Hand-derived from the definition of exact softmax attention (the pages print no "
              "numeric worked example). Each case states its derivation; values are closed forms "
              "evaluated in float64.",
    "cases": [
        {"name": "two_keys_ln3",
         "derivation": "q=[1], k=[[0],[ln 3]], scale=1: S=[0, ln3], P=[1/4, 3/4]; O=1/4*2+3/4*6=5; "
                       "L=ln(e^0+e^ln3)=ln 4. With dO=[1]: dV=P=[1/4,3/4]; dP=[2,6]; "
                       "delta=sum P*dP=5; dS=P*(dP-delta)=[-3/4,3/4]; dQ=scale*sum dS_j k_j=3/4 ln3; "
                       "dK=scale*dS*q=[-3/4,3/4].",
         "causal": False, "scale": 1.0,
         "q": [[1.0]], "k": [[0.0], [LN3]], "v": [[2.0], [6.0]], "do": [[1.0]],
         "o": [[5.0]], "lse": [math.log(4.0)],
         "dq": [[0.75 * LN3]], "dk": [[-0.75], [0.75]], "dv": [[0.25], [0.75]]},
        {"name": "causal_prefix_mean",
         "derivation": "q=0 so every visible score is 0; causal row i sees keys 0..i with equal "
                       "weight 1/(i+1): O_i = mean(v_0..v_i) = [3, 4, 6] for v=[3,5,10]; "
                       "L_i = ln(i+1).",
         "causal": True, "scale": 1.0,
         "q": [[0.0], [0.0], [0.0]], "k": [[1.0], [-2.0], [0.5]], "v": [[3.0], [5.0], [10.0]],
         "o": [[3.0], [4.0], [6.0]], "lse": [0.0, math.log(2.0), math.log(3.0)]},
        {"name": "two_dims_scale_half",
         "derivation": "D=2, scale=1/2, q=[2, 0], k=[[0,0],[ln 9, 7]]: S=[0, 1/2*2*ln9]=[0, ln 9], "
                       "P=[1/10, 9/10]; v=[[10,0],[0,10]] gives O=[1, 9]; L=ln 10.",
         "causal": False, "scale": 0.5,
         "q": [[2.0, 0.0]], "k": [[0.0, 0.0], [LN9, 7.0]], "v": [[10.0, 0.0], [0.0, 10.0]],
         "o": [[1.0, 9.0]], "lse": [math.log(10.0)]},
    ],
}

if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "handworked.json")
    with open(path, "w") as f:
        json.dump(CASES, f, indent=1)
