"""Write ``worked_example.json``: a five-node graph solved by hand.

The pages print no worked numbers for the attention aggregation, so this
fixture is a closed-form example derived by hand from the definition
(GAT additive score, Velickovic et al. 2018, eqs. 1-3; softmax over the
in-neighbours and value aggregation as in "On Efficient Scaling of GNNs via
IO-Aware Layers Implementations", Technical Summary > Methodology,
attention-based layers).  This script evaluates the hand-derived closed forms
below with ``math.exp``; it calls neither the oracle nor the CUDA path.

Instance (H = 1, D = 2, LeakyReLU slope 0.2):
  h      = (1,0) (0,1) (2,-1) (-1,3) (0.25,-2)        nodes 0..4
  a_src  = (1, 0)    -> s_src = h[:,0]   = 1, 0, 2, -1, 0.25
  a_dst  = (0, 0.5)  -> s_dst = h[:,1]/2 = 0, 0.5, -0.5, 1.5, -1
  in-neighbours: 0 <- {0, 1, 4};  1 <- {1};  2 <- {3};  3 <- {0, 0, 2} (a
  double edge);  4 <- {} (isolated)
  dout   = (1,0) (0,1) (1,1) (0,-1) (2,2)

Forward, row by row (z = s_dst(i) + s_src(j), e = z if z > 0 else 0.2 z):
  row 0: z = 1, 0, 0.25 -> e = 1, 0, 0.25;  S0 = e^1 + e^0 + e^0.25
         out0 = (e h0 + h1 + e^0.25 h4)/S0,  lse0 = ln S0
         (z = 0 exactly for the edge 1 -> 0: e = 0, and its LeakyReLU
          derivative is taken as the slope)
  row 1: one neighbour, z = 0.5:  out1 = h1,  lse1 = 0.5
  row 2: one neighbour, z = -1.5: out2 = h3,  lse2 = -0.3
  row 3: z = 2.5, 2.5, 3.5 -> alpha = (1, 1, e)/(2 + e)
         out3 = (2 h0 + e h2)/(2 + e),  lse3 = 2.5 + ln(2 + e)
  row 4: no neighbours: out4 = 0, lse4 = -inf

Backward of L = sum(out * dout), with da = dout_i . h_j, Delta_i =
sum_j alpha da, de = alpha (da - Delta_i), dz = de * LeakyReLU'(z):
  rows 1, 2: alpha = 1 so de = 0; value terms dh1 += dout1, dh3 += dout2.
  row 3: da = 0, 0, 1;  Delta3 = e/(2+e);  de = -e/(2+e)^2 (twice, source 0)
         and 2e/(2+e)^2 (source 2); all z > 0 so dz = de and ds_dst3 = 0.
         value terms: dh0 += 2/(2+e) dout3,  dh2 += e/(2+e) dout3.
  row 0: alpha = (e, 1, e^0.25)/S0;  da = 1, 0, 0.25;
         Delta0 = (e + 0.25 e^0.25)/S0;  dz_q = alpha_q (da_q - Delta0) g_q with
         g = (1, 0.2, 1);  ds_dst0 = sum_q dz_q;  ds_src gets dz_0 at node 0,
         dz_1 at node 1, dz_2 at node 4; value terms alpha_q dout0 at 0, 1, 4.
  then dh_j += ds_src(j) a_src + ds_dst(j) a_dst, da_src = sum_j ds_src(j) h_j,
  da_dst = sum_i ds_dst(i) h_i.
"""
import json
import math
import os

E = math.e


def main():
    h = [[1.0, 0.0], [0.0, 1.0], [2.0, -1.0], [-1.0, 3.0], [0.25, -2.0]]
    dout = [[1.0, 0.0], [0.0, 1.0], [1.0, 1.0], [0.0, -1.0], [2.0, 2.0]]
    a_src, a_dst, slope = [1.0, 0.0], [0.0, 0.5], 0.2
    row_ptr = [0, 3, 4, 5, 8, 8]
    col = [0, 1, 4, 1, 3, 0, 0, 2]

    e25 = math.exp(0.25)
    S0 = E + 1.0 + e25
    out = [
        [(E * 1.0 + 0.0 + e25 * 0.25) / S0, (0.0 + 1.0 + e25 * -2.0) / S0],
        [0.0, 1.0],
        [-1.0, 3.0],
        [(2.0 + 2.0 * E) / (2.0 + E), -E / (2.0 + E)],
        [0.0, 0.0],
    ]
    lse = [math.log(S0), 0.5, -0.3, 2.5 + math.log(2.0 + E), "-inf"]

    # row 0 backward pieces
    al0 = [E / S0, 1.0 / S0, e25 / S0]
    da0 = [1.0, 0.0, 0.25]
    delta0 = (E + 0.25 * e25) / S0
    g0 = [1.0, slope, 1.0]
    dz0 = [al0[q] * (da0[q] - delta0) * g0[q] for q in range(3)]
    ds_dst = [sum(dz0), 0.0, 0.0, 0.0, 0.0]
    # row 3 backward pieces
    c3 = (2.0 + E) ** 2
    ds_src = [dz0[0] - 2.0 * E / c3, dz0[1], 2.0 * E / c3, 0.0, dz0[2]]
    # value terms
    val = [[0.0, 0.0] for _ in range(5)]
    for q, j in enumerate([0, 1, 4]):
        val[j][0] += al0[q] * dout[0][0]
        val[j][1] += al0[q] * dout[0][1]
    val[1][0] += dout[1][0]; val[1][1] += dout[1][1]       # row 1, alpha = 1
    val[3][0] += dout[2][0]; val[3][1] += dout[2][1]       # row 2, alpha = 1
    val[0][0] += 2.0 / (2.0 + E) * dout[3][0]; val[0][1] += 2.0 / (2.0 + E) * dout[3][1]
    val[2][0] += E / (2.0 + E) * dout[3][0]; val[2][1] += E / (2.0 + E) * dout[3][1]
    dh = [[val[j][d] + ds_src[j] * a_src[d] + ds_dst[j] * a_dst[d] for d in range(2)]
          for j in range(5)]
    da_src = [sum(ds_src[j] * h[j][d] for j in range(5)) for d in range(2)]
    da_dst = [sum(ds_dst[j] * h[j][d] for j in range(5)) for d in range(2)]
    delta = [delta0, dout[1][1] * 1.0, dout[2][0] * -1.0 + dout[2][1] * 3.0, E / (2.0 + E), 0.0]

    fixture = dict(
        source="hand-derived closed forms; see make_worked_example.py",
        H=1, D=2, slope=slope, row_ptr=row_ptr, col_idx=col,
        h=h, a_src=a_src, a_dst=a_dst, dout=dout,
        expected=dict(out=out, lse=lse, delta=delta, ds_dst=ds_dst, ds_src=ds_src,
                      dh=dh, da_src=da_src, da_dst=da_dst),
    )
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "worked_example.json")
    with open(path, "w") as f:
        json.dump(fixture, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
