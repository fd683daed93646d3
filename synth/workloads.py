"""The five synthetic workloads (shapes, batch sizes, seeds).

Shapes follow the Kimi K3 MoE layer as the pages describe it: hidden 7168,
896 routed experts per layer of which 16 are chosen, two shared experts
(Deltafin analysis, §2.1 and §5.1; Deltafin README, "How it works"), with
MXFP4 experts of 17,547,264 bytes each (kimi-k3-in-c blog, "先把账算明白"),
which fixes the expert intermediate at 1536. The tiny workload is the
cheap correctness gate, in the spirit of kimi-k3-in-c's `make test`.
"""
from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    cfg_id: int          # folded into every generator key
    H: int               # hidden size
    I: int               # routed-expert intermediate size
    E: int               # routed experts per layer
    k: int               # experts chosen per token
    n_shared: int        # shared experts per layer
    Is: int              # intermediate size of each shared expert
    T: int               # tokens per call
    L: int = 1           # layers (stack mode when > 1)
    stack: bool = False  # RMSNorm before and residual add after each layer
    eps: float = 1e-6
    steps: int = 1       # decode steps (stack workload)
    seed: int = 0
    weights_cfg: int = -1  # generator key of the weights (-1: cfg_id)

    @property
    def wcfg(self):
        return self.cfg_id if self.weights_cfg < 0 else self.weights_cfg


K3 = dict(H=7168, I=1536, E=896, k=16, n_shared=2, Is=1536)

WORKLOADS = {
    0: Workload("tiny-h256-e8-top2", 0, H=256, I=64, E=8, k=2, n_shared=1,
                Is=64, T=1),
    1: Workload("k3-layer-decode-b1", 1, T=1, **K3),
    # batch 8 and batch 512 run on the same K3 layer as batch 1
    2: Workload("k3-layer-decode-b8", 2, T=8, weights_cfg=1, **K3),
    3: Workload("k3-layer-prefill-b512", 3, T=512, weights_cfg=1, **K3),
    4: Workload("k3-stack8-decode", 4, T=1, L=8, stack=True, steps=64, **K3),
}
