"""PowerSGD on the GPU against the oracle (binary64): the reconstruction
P_hat Q'^T and the residual within 1e-3 relative Frobenius error at every one
of several consecutive steps, plus orthonormality of P_hat."""
import numpy as np
import pytest

import oracle
from gradient_compression_ef_gb300 import inputs
from tests.gpu_helpers import dev_f32, host, torch_cuda

pytestmark = pytest.mark.gpu

TOL = 1e-3


@pytest.fixture(scope="module")
def env():
    torch = torch_cuda()
    from gradient_compression_ef_gb300 import gc
    ctx = gc.Context(1024)
    ctx.reserve_powersgd(11008, 11008, 16)
    yield torch, gc, ctx
    ctx.close()


def rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def run_steps(env, G, E, Q, r, steps):
    torch, gc, ctx = env
    m, n = G.shape
    Gd, Ed, Qd = dev_f32(torch, G), dev_f32(torch, E), dev_f32(torch, Q)
    Pd = torch.empty((m, r), dtype=torch.float32, device="cuda")
    oE, oQ = E.copy(), Q.copy()
    for s in range(steps):
        gc.powersgd_step(ctx, Gd, Ed, m, n, r, Pd, Qd)
        ctx.check()
        oP, oQ, oE = oracle.powersgd_step(G, oE, oQ, r)
        P, Qn, En = host(Pd), host(Qd), host(Ed)
        approx = P.astype(np.float64) @ Qn.astype(np.float64).T
        o_approx = oP.astype(np.float64) @ oQ.astype(np.float64).T
        assert rel(approx, o_approx) <= TOL, "step %d reconstruction" % s
        assert rel(En, oE) <= TOL * max(1.0, np.linalg.norm(o_approx) /
                                        max(np.linalg.norm(oE), 1e-30)), "step %d residual" % s
        assert np.abs(P.T.astype(np.float64) @ P - np.eye(r)).max() < 1e-4


@pytest.mark.parametrize("m,n,r", [(300, 200, 4), (257, 131, 3), (64, 1000, 1), (1000, 64, 16),
                                   (513, 515, 8), (600, 1500, 12), (700, 2052, 16),
                                   (2100, 516, 9)])
def test_small_shapes(env, m, n, r):
    M, _ = inputs.low_rank_matrix(m, n, r=r)
    rg = np.random.default_rng(m + n)
    E = (0.01 * rg.standard_normal((m, n))).astype(np.float32)
    Q = rg.standard_normal((n, r)).astype(np.float32)
    run_steps(env, M, E, Q, r, 3)


@pytest.mark.parametrize("shape", inputs.POWERSGD_SHAPES)
def test_workload_shapes_five_steps(env, shape):
    """The rank-16 + noise workload at full size, rank 4, five steps reusing Q."""
    m, n = shape
    M, Q0 = inputs.low_rank_matrix(m, n, r=4)
    run_steps(env, M, np.zeros_like(M), Q0, 4, 5)


def test_residual_matches_its_own_factors_elementwise(env):
    """E' = M - P_hat Q'^T holds element by element, with the step's own
    P_hat and Q', at every step of two five-step runs on the 4096 x 11008
    workload matrix, and Q' = M^T P_hat column by column.  A residual pass
    that read part of a staged tile after its next refill had begun gives
    wrong values in one row of a few hundred columns: far below the
    Frobenius bar of the comparisons with the oracle, but of the elements'
    own size here; the same fault in the Q' pass would move a column sum by
    one row's term of 4096 (about 1/64 of it)."""
    torch, gc, ctx = env
    m, n, r = 4096, 11008, 4
    M0, Q0 = inputs.low_rank_matrix(m, n, r=r)
    G = torch.from_numpy(M0).cuda()
    for _ in range(2):
        E = torch.zeros_like(G)
        Q = torch.from_numpy(Q0).cuda()
        P = torch.empty((m, r), dtype=torch.float32, device="cuda")
        for step in range(5):
            M = G + E  # the same binary32 sum as the step's first pass
            gc.powersgd_step(ctx, G, E, m, n, r, P, Q)
            ctx.check()
            D = E.double() - (M.double() - P.double() @ Q.double().T)
            rms = E.double().pow(2).mean().sqrt().item()
            worst = D.abs().max().item()
            assert worst <= 1e-3 * rms, "step %d: |E' - (M - P_hat Q'^T)| up to %.3e (rms %.3e)" % (
                step, worst, rms)
            del D
            Qx = M.double().T @ P.double()
            dq = (Q.double() - Qx).abs().max(dim=0).values
            scale = Qx.abs().max(dim=0).values
            assert bool((dq <= 1e-4 * scale).all()), "step %d: |Q' - M^T P_hat| / max |col| = %s" % (
                step, (dq / scale).tolist())
            del M, Qx


def test_zero_gradient(env):
    G = np.zeros((40, 36), np.float32)
    torch, gc, ctx = env
    Gd, Ed = dev_f32(torch, G), dev_f32(torch, G)
    Qd = torch.ones((36, 2), dtype=torch.float32, device="cuda")
    Pd = torch.empty((40, 2), dtype=torch.float32, device="cuda")
    gc.powersgd_step(ctx, Gd, Ed, 40, 36, 2, Pd, Qd)
    ctx.check()
    assert not host(Pd).any() and not host(Qd).any() and not host(Ed).any()


def test_requires_reserved_scratch(env):
    torch, gc, _ = env
    c = gc.Context(16)
    G = torch.zeros((8, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(gc.GCError) as ei:
        gc.powersgd_step(c, G, G.clone(), 8, 8, 2, torch.zeros((8, 2), device="cuda"),
                         torch.zeros((8, 2), device="cuda"))
    assert ei.value.status == gc.ERR_WORKSPACE
    c.close()


@pytest.mark.parametrize("shape", [(4096, 11008), (1000, 4100), (777, 96)])
def test_repeatable_and_close_to_fp32(env, shape):
    """The same step on the same inputs gives the same bits every time (the
    passes' partial sums are added in a fixed order), and the three-term
    TF32 products keep the reconstruction within 2e-5 of the binary64
    oracle -- far inside the 1e-3 bar, so that a lost or doubled partial
    sum cannot hide under it.  The shapes cover 32-column segments with a
    partial last column block (11008 = 21.5 x 512), columns that are not a
    multiple of 32 (4100) and a matrix smaller than one column block."""
    torch, gc, ctx = env
    m, n = shape
    M, Q0 = inputs.low_rank_matrix(m, n, r=4)
    outs = []
    for _ in range(2):
        Gd, Ed, Qd = dev_f32(torch, M), dev_f32(torch, np.zeros_like(M)), dev_f32(torch, Q0)
        Pd = torch.empty((m, 4), dtype=torch.float32, device="cuda")
        gc.powersgd_step(ctx, Gd, Ed, m, n, 4, Pd, Qd)
        ctx.check()
        outs.append((host(Pd), host(Qd), host(Ed)))
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    oP, oQ, oE = oracle.powersgd_step(M, np.zeros_like(M), Q0, 4)
    P, Qn, En = outs[0]
    approx = P.astype(np.float64) @ Qn.astype(np.float64).T
    o_approx = oP.astype(np.float64) @ oQ.astype(np.float64).T
    assert rel(approx, o_approx) <= 2e-5
    assert rel(En, oE) <= 2e-5 * max(1.0, np.linalg.norm(o_approx) / np.linalg.norm(oE))


@pytest.mark.parametrize("shape,r", [((1030, 2060), 16), ((777, 1540), 11)])
def test_high_rank_repeatable(env, shape, r):
    """Ranks above 8 take their own column mapping in the second pass (two
    columns per thread); the step still gives the same bits every time."""
    torch, gc, ctx = env
    m, n = shape
    M, Q0 = inputs.low_rank_matrix(m, n, r=r)
    outs = []
    for _ in range(2):
        Gd, Ed, Qd = dev_f32(torch, M), dev_f32(torch, np.zeros_like(M)), dev_f32(torch, Q0)
        Pd = torch.empty((m, r), dtype=torch.float32, device="cuda")
        gc.powersgd_step(ctx, Gd, Ed, m, n, r, Pd, Qd)
        ctx.check()
        outs.append((host(Pd), host(Qd), host(Ed)))
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("m,n,r", [(16, 100_000, 4), (40, 60_000, 16)])
def test_short_wide_matrix_in_a_tight_context(env, m, n, r):
    """Few rows and many columns, with the scratch reserved for exactly this
    shape: pass 1 then runs on more CTAs (one per SM) than the matrix has
    blocks of 8 rows, and each of them writes a Gram partial."""
    torch, gc, _ = env
    M, _ = inputs.low_rank_matrix(m, n, r=min(r, 4))
    rg = np.random.default_rng(m * n + r)
    Q = rg.standard_normal((n, r)).astype(np.float32)
    c = gc.Context(16)
    c.reserve_powersgd(m, n, r)
    try:
        run_steps((torch, gc, c), M, np.zeros_like(M), Q, r, 2)
    finally:
        c.close()


@pytest.mark.parametrize("m,n,r", [(1, 4, 1), (3, 8, 2), (17, 12, 3), (2, 1024, 2), (33, 4, 4)])
def test_tiny_shapes_on_the_tensor_core_path(env, m, n, r):
    """Rows of a 16-byte multiple (n % 4 == 0) take the tensor-core passes:
    a single row, fewer rows than one padded block of 16, four columns."""
    rg = np.random.default_rng(m * 1000 + n * 10 + r)
    G = rg.standard_normal((m, n)).astype(np.float32)
    E = (0.1 * rg.standard_normal((m, n))).astype(np.float32)
    Q = rg.standard_normal((n, r)).astype(np.float32)
    run_steps(env, G, E, Q, r, 2)
