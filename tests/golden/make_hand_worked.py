"""Writes hand_worked.json: small selective-scan cases worked out by hand.

Each expected value is the closed-form result of the derivation string stored
beside it (exact arithmetic on powers of 1/2, ln 2 and ln 3); nothing here runs
an implementation of the scan.  Run: python tests/golden/make_hand_worked.py
"""
import json
import math
import os

ln2 = math.log(2)
ln3 = math.log(3)

SCAN = [
    dict(name="one_state_three_steps",
         cite="Mamba state space model explainer (fsdata.site), section 3.2, selective_step",
         derivation="softplus off, Delta_raw=1, bias=0 so Delta=1; A=-ln2 so A_bar=exp(-ln2)=1/2; B_bar=Delta*B=2. "
                    "h0=0.5*0+2*1=2, y0=2+0.5*1=2.5; h1=0.5*2+2*3=7, y1=7+0.5*3=8.5; "
                    "h2=0.5*7+2*(-2)=-0.5, y2=-0.5+0.5*(-2)=-1.5",
         N=1, L=3, softplus=0, A=[[-ln2]], delta=[1, 1, 1], bias=0.0, B=[[2, 2, 2]], C=[[1, 1, 1]], D=0.5,
         u=[1, 3, -2], z=None, zoh=0, y=[2.5, 8.5, -1.5], last=[-0.5]),
    dict(name="two_states_softplus_at_zero",
         cite="Mamba state space model explainer (fsdata.site), section 3.2; softplus(0)=ln 2",
         derivation="softplus on, Delta_raw=0, bias=0 so Delta=ln2; A=(-1,0) so A_bar=(exp(-ln2), exp(0))=(1/2,1); "
                    "B=(1,1), C=(1,2), D=0. t0: h=(ln2*2, ln2*2), y0=2ln2+2*2ln2=6ln2; "
                    "t1: h=(0.5*2ln2+4ln2, 2ln2+4ln2)=(5ln2,6ln2), y1=5ln2+12ln2=17ln2",
         N=2, L=2, softplus=1, A=[[-1.0, 0.0]], delta=[0, 0], bias=0.0, B=[[1, 1], [1, 1]], C=[[1, 1], [2, 2]],
         D=0.0, u=[2, 4], z=None, zoh=0, y=[6 * ln2, 17 * ln2], last=[5 * ln2, 6 * ln2]),
    dict(name="one_state_gated",
         cite="Mamba tutorial (freeguideonline) section 4.1 and the PyTorch block of the ai.xwebgame summary: "
              "output times SiLU(z)",
         derivation="the case one_state_three_steps with z=(0, ln3, -ln3); SiLU(0)=0, SiLU(ln3)=ln3/(1+1/3)=0.75ln3, "
                    "SiLU(-ln3)=-ln3/(1+3)=-0.25ln3; y=(2.5*0, 8.5*0.75ln3, -1.5*(-0.25ln3))",
         N=1, L=3, softplus=0, A=[[-ln2]], delta=[1, 1, 1], bias=0.0, B=[[2, 2, 2]], C=[[1, 1, 1]], D=0.5,
         u=[1, 3, -2], z=[0.0, ln3, -ln3], zoh=0, y=[0.0, 8.5 * 0.75 * ln3, 0.375 * ln3], last=[-0.5]),
    dict(name="one_state_bias_no_softplus",
         cite="Mamba tutorial (freeguideonline) section 4.2 step 2 (Delta bias); "
              "reading: with softplus off Delta = Delta_raw + bias",
         derivation="softplus off, Delta_raw=(0.5,0.5), bias=0.5 so Delta=1; A=-ln2 so A_bar=1/2; B=1, C=3, D=0, "
                    "u=(4,4). h0=4, y0=12; h1=0.5*4+4=6, y1=18",
         N=1, L=2, softplus=0, A=[[-ln2]], delta=[0.5, 0.5], bias=0.5, B=[[1, 1]], C=[[3, 3]], D=0.0, u=[4, 4],
         z=None, zoh=0, y=[12.0, 18.0], last=[6.0]),
    dict(name="one_state_zoh",
         cite="Mamba tutorial (freeguideonline) section 2.2, zero-order hold "
              "B_bar=(Delta A)^-1 (exp(Delta A)-I) Delta B",
         derivation="Delta=1, A=-ln2: A_bar=1/2, B_bar=(1/2-1)/(-ln2)*B = B/(2ln2) = 1/ln2 for B=2; C=1, D=0, "
                    "u=(1,1). h0=1/ln2=y0; h1=0.5/ln2+1/ln2=1.5/ln2=y1",
         N=1, L=2, softplus=0, A=[[-ln2]], delta=[1, 1], bias=0.0, B=[[2, 2]], C=[[1, 1]], D=0.0, u=[1, 1],
         z=None, zoh=1, y=[1 / ln2, 1.5 / ln2], last=[1.5 / ln2]),
]

STEP = [
    dict(name="decode_one_step",
         cite="Mamba state space model explainer (fsdata.site), section 3.2, selective_step applied to a stored state",
         derivation="state=(1,-1), softplus off, Delta=1, A=(-ln2,-ln2) so A_bar=1/2; B=(1,2), u=2 so "
                    "B_bar*u=(2,4); h=(0.5+2, -0.5+4)=(2.5,3.5); C=(1,1), D=1: y=2.5+3.5+1*2=8",
         N=2, softplus=0, state=[1.0, -1.0], A=[-ln2, -ln2], delta=1.0, bias=0.0, B=[1, 2], C=[1, 1], D=1.0,
         u=2.0, z=None, y=8.0, new_state=[2.5, 3.5]),
]

if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "hand_worked.json")
    with open(out, "w") as f:
        json.dump(dict(note="hand-derived worked cases of the selective scan; expected values follow from the "
                            "derivation text, not from running any implementation", scan=SCAN, step=STEP),
                  f, indent=1)
