"""The Python binding validates every tensor before a pointer reaches the
C-ABI (CPU only): wrong shapes, dtypes, devices or layouts raise instead of
handing the library a host pointer or a short buffer.  The graph here is a
stand-in that only carries what the checks read (its device and N); every
call below must fail before the library is touched."""
import pytest
import torch

import graph_neural_network_gb300 as gnn


class _FakeGraph:
    def __init__(self, n):
        self.n = n
        self.device = torch.device("cuda", 0)

    @property
    def _lib(self):
        raise AssertionError("the library was reached before the arguments were checked")


N, H, D = 6, 2, 8
G = _FakeGraph(N)


def _feat(*shape, dtype=torch.float32):
    return torch.zeros(*shape, dtype=dtype)


@pytest.mark.parametrize("h, err", [
    (_feat(N, H), ValueError),                       # not [N, H, D]
    (_feat(N + 1, H, D), ValueError),                # wrong N
    (_feat(N, H, D, dtype=torch.float64), TypeError),
    (_feat(N, H, D), ValueError),                    # a host tensor
])
def test_gat_forward_rejects_bad_features(h, err):
    with pytest.raises(err):
        gnn.gat_forward(G, h, _feat(H, D), _feat(H, D), 0.2)


def test_attention_vectors_are_checked():
    h = _feat(N, H, D)
    for a, err in ((_feat(D), ValueError), (_feat(H, D + 1), ValueError),
                   (torch.zeros(H, D, dtype=torch.int32), TypeError), (_feat(H, D), ValueError)):
        with pytest.raises(err):
            gnn._att(G, a, "a_src", H, D)
    with pytest.raises(TypeError):
        gnn._att(G, [[0.0] * D] * H, "a_src", H, D)


def test_supplied_outputs_are_checked():
    for t, shape, dtype, err in (
            (_feat(N - 1, H, D), (N, H, D), torch.float32, ValueError),    # short out
            (_feat(N, H), (N, H), torch.bfloat16, TypeError),             # wrong dtype
            (_feat(N, H), (N, H), torch.float32, ValueError),             # host lse
            (_feat(H, D).t(), (D, H), torch.float32, ValueError)):        # host, strided
        with pytest.raises(err):
            gnn._given(G, t, "out", shape, dtype, lambda: None)
    assert gnn._given(G, None, "out", (1,), torch.float32, lambda: "made") == "made"


def test_workspace_is_checked():
    with pytest.raises(TypeError):
        gnn._check_ws(G, torch.zeros(64, dtype=torch.float32))
    with pytest.raises(ValueError):
        gnn._check_ws(G, torch.zeros(64, dtype=torch.uint8))        # host memory
    assert gnn._check_ws(G, None) is None


def test_other_families_check_their_inputs():
    x2 = _feat(N, H * D)
    with pytest.raises(ValueError):
        gnn.gcn_forward(G, x2, "sym")                   # host features
    with pytest.raises(ValueError):
        gnn.gcn_forward(G, _feat(N + 2, 4), "sym")      # wrong N
    with pytest.raises(ValueError):
        gnn.reduce_forward(G, x2, "max")
    with pytest.raises(ValueError):
        gnn.gatv2_forward(G, _feat(N, H, D), _feat(N, H, D), _feat(H, D), 0.2)
    with pytest.raises(ValueError):
        gnn.transformer_forward(G, _feat(N, H, D), _feat(N, H, D), _feat(N, H, D))
    with pytest.raises(ValueError):
        gnn.gat_backward(G, _feat(N, H, D), _feat(H, D), _feat(H, D), 0.2, _feat(N, H),
                         _feat(N, H, D))
