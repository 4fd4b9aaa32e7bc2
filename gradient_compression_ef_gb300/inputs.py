"""Seeded synthetic inputs shaped like the workloads the pages describe.

This module draws random numbers and lays out buffers; it holds none of the
compressor's arithmetic.  Both the CUDA path and the CPU oracle consume the
arrays it returns, so both sides always see identical bytes.

Workloads (the pages name no public dataset; every input is synthetic):

* ``demo_gradient`` -- the Python demo of "梯度聚合通信优化实战方案"
  (section Python 演示): one million N(0, 1) float32 values from
  ``numpy.random.default_rng(42)``.
* ``correlated_steps`` / ``bucket_bounds`` -- a flat float32 gradient cut
  into 25 MiB buckets (6,553,600 elements; "梯度聚合通信优化实战方案",
  通信计算重叠: buckets of 5-25 MB), Student-t (nu = 3) values times 1e-3,
  and temporally correlated steps g_t = 0.9 g_{t-1} + 0.436 fresh_t.
* ``outlier_gradient`` -- N(0, 0.01^2) with 0.1 % of the positions (distinct,
  random) multiplied by 100, for group-wise quantisation.
* ``transformer_tensor`` -- one tensor of a 32-layer transformer gradient set
  {4096x4096 x4, 4096x11008 x2, 11008x4096, 4096}, N(0, (1e-3/sqrt(fan_in))^2)
  with fan_in the first dimension.
* ``low_rank_matrix`` -- a rank-16 matrix with singular values 0.05^(i/15),
  i = 0..15 (1 down to 0.05), plus N(0, 1e-4^2) noise, and a N(0, 1) start Q.
"""
import numpy as np

BUCKET_BYTES = 25 * 1024 * 1024
BUCKET_ELEMS = BUCKET_BYTES // 4          # 6,553,600 float32 per bucket
FLAT_ELEMS = 134_217_728                  # 512 MiB flat gradient
GROUP_ELEMS = 1 << 30                     # group-wise quantisation workload

TRANSFORMER_LAYERS = 32
# (rows, cols) of the tensors of one layer: 4 attention projections, the
# two up projections, the down projection and one norm vector.
TRANSFORMER_SHAPES = ((4096, 4096),) * 4 + ((4096, 11008),) * 2 + \
    ((11008, 4096), (4096,))
POWERSGD_SHAPES = ((4096, 4096), (4096, 11008), (11008, 4096))


def rng(seed):
    return np.random.default_rng(seed)


def demo_gradient(n=1_000_000, seed=42):
    """N(0, 1) float32, the demo's simulate_gradients recipe."""
    return rng(seed).standard_normal(n).astype(np.float32)


def ratio_k(n, num, den):
    """k = max(1, floor(n * num / den)) in exact integer arithmetic
    ("4、梯度累积与梯度压缩" 4.2.1 takes k = max(1, int(n * ratio)))."""
    return max(1, (n * num) // den) if n > 0 else 0


def student_t(generator, n, nu=3, scale=1e-3):
    """Student-t draws Z / sqrt(V / nu) in float32, where V is a chi-square
    with integer nu degrees of freedom built as a sum of nu squared normals."""
    z = generator.standard_normal(n, dtype=np.float32)
    v = np.zeros(n, dtype=np.float32)
    for _ in range(int(nu)):
        w = generator.standard_normal(n, dtype=np.float32)
        w *= w
        v += w
    v *= np.float32(1.0 / nu)
    np.sqrt(v, out=v)
    z /= v
    z *= np.float32(scale)
    return z


def student_t_device(n, device, seed, nu=3, scale=1e-3):
    """The same Student-t recipe drawn by torch on ``device`` (seeded),
    for workloads too large to draw on the host quickly."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    z = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
    v = torch.zeros(n, device=device, dtype=torch.float32)
    for _ in range(int(nu)):
        w = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
        v.addcmul_(w, w)
    v.mul_(1.0 / nu).sqrt_()
    return z.div_(v).mul_(scale)


def correlated_steps_device(n, steps, device, seed=42, rho=0.9, fresh=0.436):
    """List of ``steps`` correlated gradients drawn by torch on ``device``."""
    out = [student_t_device(n, device, seed)]
    for t in range(1, steps):
        g = out[-1] * rho
        g.add_(student_t_device(n, device, seed * 1000 + t), alpha=fresh)
        out.append(g)
    return out


def correlated_steps(n=FLAT_ELEMS, steps=10, seed=42, rho=0.9, fresh=0.436):
    """Yields ``steps`` float32 gradients g_t = rho g_{t-1} + fresh * t-noise.

    g_0 is plain t-noise.  Each yielded array is a new buffer."""
    generator = rng(seed)
    g = student_t(generator, n)
    yield g.copy()
    for _ in range(1, steps):
        g *= np.float32(rho)
        noise = student_t(generator, n)
        noise *= np.float32(fresh)
        g += noise
        yield g.copy()


def bucket_bounds(n=FLAT_ELEMS, bucket=BUCKET_ELEMS):
    """[(start, length)] of consecutive buckets; the last may be partial."""
    return [(s, min(bucket, n - s)) for s in range(0, n, bucket)]


def outlier_gradient(n=GROUP_ELEMS, seed=42, std=0.01, frac=0.001, mult=100.0):
    """N(0, std^2) float32 with round(frac * n) distinct positions x mult."""
    generator = rng(seed)
    x = generator.standard_normal(n, dtype=np.float32)
    x *= np.float32(std)
    m = int(round(frac * n))
    if m > 0:
        pos = np.unique(generator.integers(0, n, size=m + m // 8 + 16))
        generator.shuffle(pos)
        pos = pos[:m]
        x[pos] *= np.float32(mult)
    return x


def outlier_gradient_device(n, device, seed, std=0.01, frac=0.001, mult=100.0):
    """The outlier recipe drawn by torch on ``device`` (seeded): N(0, std^2)
    with round(frac * n) distinct positions (a random permutation's prefix)
    multiplied by mult."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    x = torch.randn(n, generator=gen, device=device, dtype=torch.float32).mul_(std)
    m = int(round(frac * n))
    if m > 0:
        pos = torch.randperm(n, generator=gen, device=device)[:m]
        x[pos] *= mult
    return x


def transformer_tensor_device(layer, which, device, seed=42, scale=1e-3):
    """Tensor ``which`` of ``layer`` with the same distribution as
    transformer_tensor, drawn by torch on ``device`` (seeded)."""
    import torch
    shape = TRANSFORMER_SHAPES[which]
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) * 1_000_003 + int(layer) * 1009 + int(which))
    n = int(np.prod(shape))
    return torch.randn(n, generator=gen, device=device,
                       dtype=torch.float32).mul_(scale / float(np.sqrt(shape[0])))


def transformer_set_sizes(layers=TRANSFORMER_LAYERS):
    """[(elements, fan_in)] of every tensor of the layer set, layer by layer."""
    one = [(int(np.prod(s)), s[0]) for s in TRANSFORMER_SHAPES]
    return one * int(layers)


def transformer_set_device(layers, steps, device, seed=42, scale=1e-3, rho=0.9, fresh=0.436):
    """``steps`` flat float32 gradients of the whole layer set (tensors laid
    end to end, layer by layer), drawn by torch on ``device`` (seeded).
    Tensor t of step 0 is N(0, (scale / sqrt(fan_in_t))^2); later steps are
    temporally correlated, g_s = rho g_{s-1} + fresh * (a new draw of the
    same distribution), so each tensor keeps its distribution (rho^2 +
    fresh^2 = 1.0001)."""
    import torch
    sizes = transformer_set_sizes(layers)
    total = sum(n for n, _ in sizes)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))

    def draw():
        x = torch.randn(total, generator=gen, device=device, dtype=torch.float32)
        a = 0
        for n, fan_in in sizes:
            x[a:a + n].mul_(scale / float(np.sqrt(fan_in)))
            a += n
        return x

    out = [draw()]
    for _ in range(1, steps):
        g = draw().mul_(fresh)
        g.add_(out[-1], alpha=rho)
        out.append(g)
    return out


def transformer_tensor(layer, which, seed=42, scale=1e-3):
    """Tensor ``which`` (0..7) of ``layer`` as a flat float32 array."""
    shape = TRANSFORMER_SHAPES[which]
    fan_in = shape[0]
    generator = rng([seed, layer, which])
    n = int(np.prod(shape))
    x = generator.standard_normal(n, dtype=np.float32)
    x *= np.float32(scale / np.sqrt(fan_in))
    return x


def low_rank_matrix(m, n, rank=16, noise_std=1e-4, seed=42, r=4):
    """(M float32 m x n, Q0 float32 n x r) for the PowerSGD workload.

    M = U diag(sigma) V^T + noise with U, V orthonormal (QR of seeded
    Gaussians) and sigma_i = 0.05^(i / (rank - 1))."""
    generator = rng([seed, m, n])
    u, _ = np.linalg.qr(generator.standard_normal((m, rank)))
    v, _ = np.linalg.qr(generator.standard_normal((n, rank)))
    sigma = 0.05 ** (np.arange(rank) / max(rank - 1, 1))
    M = (u * sigma) @ v.T
    M = M.astype(np.float32)
    M += generator.standard_normal((m, n), dtype=np.float32) * \
        np.float32(noise_std)
    Q0 = generator.standard_normal((n, r), dtype=np.float32)
    return M, Q0


def low_rank_matrix_device(m, n, device, seed=42, rank=16, noise_std=1e-4, r=4):
    """The low_rank_matrix recipe with the large parts drawn by torch on
    ``device`` (seeded): (M float32 m x n, Q0 float32 n x r) with M = U
    diag(sigma) V^T + noise, U, V orthonormal (numpy QR of Gaussians),
    sigma_i = 0.05^(i / (rank - 1)) -- the same distribution as the host
    recipe, for workloads too large to draw on the host."""
    import torch
    # the thin orthonormal factors come from numpy's QR on the host (small)
    generator = rng([seed, m, n, 1])
    u, _ = np.linalg.qr(generator.standard_normal((m, rank)))
    v, _ = np.linalg.qr(generator.standard_normal((n, rank)))
    sigma = 0.05 ** (np.arange(rank) / max(rank - 1, 1))
    u = torch.from_numpy(u * sigma).to(device)
    v = torch.from_numpy(v).to(device)
    M = (u @ v.T).to(torch.float32)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    M.add_(torch.randn(m, n, generator=gen, device=device, dtype=torch.float32),
           alpha=noise_std)
    Q0 = torch.randn(n, r, generator=gen, device=device, dtype=torch.float32)
    return M, Q0


def tiny_cases(seed=7):
    """Small edge-case vectors used by the parity tests (length, values)."""
    generator = rng(seed)
    cases = []
    for n in (1, 2, 3, 4, 5, 7, 8, 63, 64, 65, 127, 128, 129, 255, 1000, 4097):
        cases.append(("normal_%d" % n,
                      generator.standard_normal(n).astype(np.float32)))
    cases.append(("all_equal", np.full(777, 0.25, dtype=np.float32)))
    cases.append(("zeros", np.zeros(300, dtype=np.float32)))
    cases.append(("signed_zeros",
                  np.array([0.0, -0.0] * 70, dtype=np.float32)))
    cases.append(("few_levels",
                  generator.integers(-3, 4, size=2049).astype(np.float32)))
    cases.append(("one_outlier",
                  np.concatenate([np.full(513, 1e-3, np.float32),
                                  np.array([50.0], np.float32)])))
    return cases
